"""The C ABI on the host, no GPU: the library loads, exports every function the
header declares, and rejects bad arguments with the documented status codes
before making any CUDA call."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_router.h")


@pytest.fixture(scope="module")
def lib():
    from top_gating_expert_row_gb300 import build

    build.build()
    import top_gating_expert_row_gb300 as m

    return m


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"\b(moe_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = _declared()
    for want in ("moe_router_fwd", "moe_router_bwd", "moe_aux_scores_fwd", "moe_aux_scores_bwd", "moe_sort",
                 "moe_sort_capacity", "moe_sort_workspace_bytes", "moe_router_fused_fwd_sort",
                 "moe_router_fused_workspace_bytes", "moe_router_strerror"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", lib.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r" T (\w+)$", out, re.M))
    missing = [n for n in _declared() if n not in exported]
    assert not missing, missing
    cdll = ctypes.CDLL(lib.LIB_PATH)
    for n in _declared():
        assert getattr(cdll, n) is not None


def test_binding_wraps_every_symbol(lib):
    for n in _declared():
        assert callable(getattr(lib, n)), n


def test_strerror(lib):
    for code in (0, 1, 2, 3, 4, 5):
        assert lib.strerror(code).startswith("MR_")
    assert (lib.MR_ERANGE, lib.MR_ETIMEOUT) == (4, 5)
    assert "unknown" in lib.strerror(99)


def test_device_status_rejects_null_output(lib):
    assert lib._lib.moe_router_device_status(None, 0, None) == lib.MR_EINVAL


def _p(lib, **kw):
    base = dict(T=4, E=64, topk=4)
    base.update(kw)
    return lib.RouterParams(**base)


FAKE = 0x10000  # never dereferenced: every call below fails validation first


def _fwd(lib, p, logits=FAKE, probs=FAKE):
    cp = p.c()
    return lib._lib.moe_router_fwd(ctypes.byref(cp), logits, probs, None, None, None, None, None, None)


@pytest.mark.parametrize("kw,code", [
    (dict(E=0), 1), (dict(T=-1), 1), (dict(topk=0), 1), (dict(topk=65), 1),
    (dict(score_fn=2), 1), (dict(in_dtype=5), 1), (dict(n_shared=4), 1), (dict(n_shared=-1), 1),
    (dict(n_group=3, topk_group=1, score_fn=1), 1),           # E % n_group != 0
    (dict(n_group=4, topk_group=5, score_fn=1), 1),           # topk_group > n_group
    (dict(n_group=4, topk_group=3, score_fn=1), 1),           # k_r % topk_group != 0
    (dict(n_group=32, topk_group=1, topk=4, score_fn=1), 1),  # k_r/topk_group > E/n_group
    (dict(T=1 << 20, E=2048), 1),                             # T*E > INT_MAX
    (dict(E=9000, topk=8), 2),                                # beyond MR_MAX_EXPERTS (8192)
    (dict(E=512, topk=300), 2),                               # k_r beyond MR_MAX_TOPK
    (dict(n_group=64, topk_group=2, E=128, score_fn=1), 2),   # more groups than lanes
    (dict(E=256, topk=32, n_group=2, topk_group=2, score_fn=1), 2),  # 16 keys per group score
    (dict(n_group=4, topk_group=2), 2),                       # softmax with groups
])
def test_fwd_rejects(lib, kw, code):
    assert _fwd(lib, _p(lib, **kw)) == code


def test_fwd_rejects_bias_with_softmax_and_missing_pointers(lib):
    p = _p(lib)
    cp = p.c()
    cp.bias = FAKE
    assert lib._lib.moe_router_fwd(ctypes.byref(cp), FAKE, FAKE, None, None, None, None, None, None) == 2
    assert _fwd(lib, _p(lib), logits=None) == 1
    assert _fwd(lib, _p(lib), probs=None) == 1  # no output at all
    assert lib._lib.moe_router_fwd(None, FAKE, FAKE, None, None, None, None, None, None) == 1


def test_zero_tokens_is_a_no_op(lib):
    assert _fwd(lib, _p(lib, T=0)) == 0
    cp = _p(lib, T=0).c()
    assert lib._lib.moe_router_bwd(ctypes.byref(cp), FAKE, FAKE, FAKE, FAKE, None) == 0
    assert lib._lib.moe_aux_scores_fwd(0, 64, 4, 0, 0, FAKE, FAKE, None, None) == 0
    assert lib._lib.moe_aux_scores_bwd(0, 64, 0, FAKE, FAKE, FAKE, None) == 0


def test_bwd_and_aux_reject(lib):
    cp = _p(lib).c()
    assert lib._lib.moe_router_bwd(ctypes.byref(cp), None, FAKE, FAKE, FAKE, None) == 1
    assert lib._lib.moe_router_bwd(ctypes.byref(cp), FAKE, FAKE, None, FAKE, None) == 1
    cp = _p(lib, E=9000).c()
    assert lib._lib.moe_router_bwd(ctypes.byref(cp), FAKE, FAKE, FAKE, FAKE, None) == 2
    assert lib._lib.moe_aux_scores_fwd(4, 64, 65, 0, 0, FAKE, FAKE, None, None) == 1
    assert lib._lib.moe_aux_scores_fwd(4, 64, 4, 0, 0, FAKE, None, None, None) == 1
    assert lib._lib.moe_aux_scores_bwd(4, 64, 3, FAKE, FAKE, FAKE, None) == 1


def test_sort_sizes_and_rejects(lib):
    assert lib.moe_sort_capacity(16, 2, 8, 4) == 32 + 8 * 3
    assert lib.moe_sort_capacity(16384, 9, 385, 64) == 147456 + 385 * 63
    assert lib.moe_sort_capacity(1, 8, 256, 32) == 8 + 8 * 31
    assert lib.moe_sort_workspace_bytes(16384, 9, 385, 64) >= 385 * 4
    assert lib.moe_sort_workspace_bytes(4, 2, 8, 0) == 0
    s = lib._lib.moe_sort
    args = [FAKE, FAKE, 4, 2, 8, 4, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 20, None, None]

    def call(**over):
        a = list(args)
        pos = dict(idx=0, T=2, topk=3, E_tot=4, bm=5, ids=6, eids=8, npp=9, ws=10, wsb=11)
        for k, v in over.items():
            a[pos[k]] = v
        return s(*a)

    assert call(T=-1) == 1 and call(topk=0) == 1 and call(E_tot=0) == 1 and call(bm=0) == 1
    assert call(ids=None) == 1 and call(eids=None) == 1 and call(npp=None) == 1
    assert call(idx=None) == 1
    # up to 4096 pairs one CTA sorts without a workspace; above that the
    # workspace holds per-chunk prefixes and cluster totals
    assert lib.moe_sort_workspace_bytes(4, 2, 8, 4) == 0
    assert lib.moe_sort_workspace_bytes(2048, 2, 8, 4) == 0
    assert lib.moe_sort_workspace_bytes(2049, 2, 8, 4) > 0
    assert call(T=4096, ws=None) == 1             # workspace needed, none given
    assert call(T=4096, wsb=0) == 1               # workspace too small
    assert call(E_tot=5000) == 2                  # beyond MR_MAX_SORT_EXPERTS
    assert call(T=1 << 28, topk=16) == 1          # T*topk >= INT_MAX


def test_wide_rows_accepted_up_to_the_limit(lib):
    # rows up to 8192 experts are routed (held in shared memory); their sort is
    # limited to 4096 experts, so the fused call refuses wider rows
    assert lib.moe_router_fused_workspace_bytes(_p(lib, T=100, E=8192, topk=8), 8) == 0
    assert lib.moe_router_fused_workspace_bytes(_p(lib, T=100, E=4096, topk=8), 8) > 0
    cp = _p(lib, T=100, E=8160, topk=8).c()
    f = lib._lib.moe_router_fused_fwd_sort
    assert f(ctypes.byref(cp), FAKE, 8, None, None, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 30, None, None) == 2


def test_fused_rejects(lib):
    cp = _p(lib, T=65).c()
    f = lib._lib.moe_router_fused_fwd_sort
    assert f(ctypes.byref(cp), FAKE, 0, None, None, FAKE, FAKE, FAKE, FAKE, None, 0, None, None) == 1
    assert f(ctypes.byref(cp), FAKE, 8, None, None, None, FAKE, FAKE, FAKE, None, 0, None, None) == 1
    # above the one-launch sizes a workspace is needed
    assert lib.moe_router_fused_workspace_bytes(_p(lib, T=65), 8) > 0
    assert f(ctypes.byref(cp), FAKE, 8, None, None, FAKE, FAKE, FAKE, FAKE, None, 0, None, None) == 1
    assert lib.moe_router_fused_workspace_bytes(_p(lib, T=17, E=512), 8) > 0
    # one launch: T <= 16 for E <= 1024, T <= 64 for E <= 256
    assert lib.moe_router_fused_workspace_bytes(_p(lib, T=16, E=1024, topk=8), 8) == 0
    assert lib.moe_router_fused_workspace_bytes(_p(lib, T=64, E=256, topk=8), 8) == 0
    assert lib.moe_router_fused_workspace_bytes(_p(lib, T=64), 8) == 0


def test_noalloc_scratch_size_matches_the_header(lib):
    text = open(HEADER).read()
    m = re.search(r"#define\s+MR_SORT_NOALLOC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", text)
    assert m, "MR_SORT_NOALLOC_SCRATCH_BYTES not found in the header"
    assert lib.moe_sort_noalloc_scratch_bytes() == int(m.group(1)) << int(m.group(2))


def test_set_launch_overlap(lib):
    assert lib._lib.moe_router_set_launch_overlap(2) == lib.MR_EINVAL
    assert lib._lib.moe_router_set_launch_overlap(-1) == lib.MR_EINVAL
    assert lib._lib.moe_router_set_launch_overlap(0) == lib.MR_OK
    assert lib._lib.moe_router_set_launch_overlap(1) == lib.MR_OK


def test_set_wait_test(lib):
    assert lib._lib.moe_router_set_wait_test(4, 2) == lib.MR_EINVAL
    assert lib._lib.moe_router_set_wait_test(4, -1) == lib.MR_EINVAL
    assert lib._lib.moe_router_set_wait_test(0, 0) == lib.MR_OK


def test_set_topk_path(lib):
    assert lib._lib.moe_router_set_topk_path(-1, 0) == 1
    assert lib._lib.moe_router_set_topk_path(8, 3) == 1
    assert lib._lib.moe_router_set_topk_path(8, 0) == 0
    assert lib._lib.moe_router_expf(None, None, -1, None) == 1
    assert lib._lib.moe_router_expf(None, None, 0, None) == 0


def test_bwd_dtype_rejects(lib):
    cp = _p(lib).c()
    f = lib._lib.moe_router_bwd_dtype
    assert f(ctypes.byref(cp), 5, FAKE, FAKE, FAKE, FAKE, None) == lib.MR_EINVAL
    assert f(ctypes.byref(cp), lib.MR_BF16, None, FAKE, FAKE, FAKE, None) == lib.MR_EINVAL
    assert f(ctypes.byref(cp), lib.MR_BF16, FAKE, FAKE, FAKE, None, None) == lib.MR_EINVAL
    assert f(ctypes.byref(_p(lib, E=9000).c()), lib.MR_BF16, FAKE, FAKE, FAKE, FAKE, None) == lib.MR_EUNSUPPORTED
    assert f(ctypes.byref(_p(lib, T=0).c()), lib.MR_BF16, FAKE, FAKE, FAKE, FAKE, None) == lib.MR_OK


def test_aux_loss_sizes_and_rejects(lib):
    L = lib._lib
    assert L.moe_aux_loss_workspace_bytes(0, 64) == 0
    assert L.moe_aux_loss_workspace_bytes(-1, 64) == 0
    # per-chunk column sums (256 rows per chunk, at most 256 chunks), one fp64 per
    # 128-column slab, and a counter
    assert L.moe_aux_loss_workspace_bytes(8192, 2304) == 32 * 2304 * 4 + 18 * 8 + 16
    assert L.moe_aux_loss_workspace_bytes(10 ** 6, 64) == 256 * 64 * 4 + 1 * 8 + 16
    ws = L.moe_aux_loss_workspace_bytes(100, 8)
    ok = dict(T=100, E=8, topk=2, coeff=0.1, N=100, probs=FAKE, tpe=FAKE, loss=FAKE, ws=FAKE, wsb=ws)

    def fwd(**kw):
        a = dict(ok, **kw)
        return L.moe_aux_loss_fwd(a["T"], a["E"], a["topk"], a["coeff"], a["N"], a["probs"], a["tpe"], a["loss"],
                                  a["ws"], a["wsb"], None)

    for bad in (dict(T=-1), dict(E=0), dict(topk=0), dict(N=0), dict(probs=None), dict(tpe=None), dict(loss=None),
                dict(ws=None), dict(wsb=ws - 1), dict(T=1 << 20, E=4096), dict(ws=FAKE + 8)):
        assert fwd(**bad) == lib.MR_EINVAL, bad
    assert L.moe_aux_loss_bwd(100, 8, 2, 0.1, 0, FAKE, FAKE, FAKE, None) == lib.MR_EINVAL
    assert L.moe_aux_loss_bwd(100, 8, 2, 0.1, 100, None, FAKE, FAKE, None) == lib.MR_EINVAL
    assert L.moe_aux_loss_bwd(100, 8, 2, 0.1, 100, FAKE, None, FAKE, None) == lib.MR_EINVAL
    assert L.moe_aux_loss_bwd(100, 8, 2, 0.1, 100, FAKE, FAKE, None, None) == lib.MR_EINVAL
    assert L.moe_tokens_per_expert(100, 8, None, FAKE, None) == lib.MR_EINVAL
    assert L.moe_tokens_per_expert(100, 8, FAKE, None, None) == lib.MR_EINVAL
    assert L.moe_tokens_per_expert(-1, 8, FAKE, FAKE, None) == lib.MR_EINVAL
