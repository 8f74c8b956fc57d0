"""GPU parity of the router forward / backward and the aux-loss scores against
the CPU oracle, through the C ABI. Both top-k paths (repeated arg-max and
threshold-select) are run on every case and must agree with the oracle, and
therefore with each other, bit for bit on indices and routing maps."""
import numpy as np
import pytest
import torch

import synth
from parity import assert_bf16_close, assert_close, assert_equal, note_near_ties, sample_rows

pytestmark = pytest.mark.gpu

SM, SG = synth.SOFTMAX, synth.SIGMOID
F32, BF16 = synth.F32, synth.BF16
ARGMAX, SELECT = 1, 2


def W(name, T, E, k, fn=SM, dt=F32, **kw):
    return synth.Workload(name, T, E, k, fn, dt, **kw)


# Oracle-sized cases: several CTAs' worth of rows, ragged tails, every row width.
CASES = [
    synth.tiny(),
    W("e64_k4", 1000, 64, 4),
    W("e256_k8_bf16_renorm", 777, 256, 8, SM, BF16, renorm=1),
    W("e384_grouped_shared_bf16", 513, 384, 9, SG, BF16, renorm=1, scaling=2.827, n_group=8,
      topk_group=4, n_shared=1, bias_range=0.05, zipf_s=1.1),
    W("e512_k4_sigma2", 300, 512, 4, sigma=2.0),
    W("e512_k8_sigma2", 300, 512, 8, sigma=2.0),
    W("e512_k22_sigma2", 300, 512, 22, sigma=2.0),
    W("e512_k36_sigma2", 300, 512, 36, sigma=2.0),
    W("e2304_k36_softmax", 200, 2304, 36),
    W("e2304_k36_sigmoid_bias", 200, 2304, 36, SG, renorm=1, scaling=2.5, bias_range=0.1),
    W("e100_k5_sigmoid_scalar_path", 100, 100, 5, SG),
    W("e37_k3_softmax_scalar_path", 64, 37, 3),
    W("e130_k7_sigmoid_bias", 50, 130, 7, SG, bias_range=0.1),
    W("e1000_k20_sigmoid_renorm", 33, 1000, 20, SG, renorm=1, scaling=1.5),
    W("e768_k64", 40, 768, 64, sigma=0.5),
    W("e1536_k100_sigmoid", 20, 1536, 100, SG, renorm=1),
    W("e24_k24_sigmoid_all", 20, 24, 24, SG, scaling=3.0),
    W("e8_k8_softmax_all", 9, 8, 8, renorm=1),
    W("e256_g16_k4_m1", 100, 256, 4, SG, renorm=1, n_group=16, topk_group=4, bias_range=0.01),
    W("e192_g4_k8_m4", 70, 192, 8, SG, renorm=1, n_group=4, topk_group=2, n_shared=2, shared_weight=0.5),
    W("e48_g3_k6_m2", 70, 48, 6, SG, n_group=3, topk_group=3),
    W("bf16_e2304_k36", 64, 2304, 36, SM, BF16),
    W("e64_k4_bf16", 200, 64, 4, SM, BF16),
    W("e100_k37_bf16_ragged", 80, 100, 37, SM, BF16, renorm=1),
    W("e768_k40_bf16", 60, 768, 40, SM, BF16, sigma=0.5),
    # rows wider than the register-resident buckets, up to the library's limit
    W("e4096_k36", 64, 4096, 36),
    W("e5000_k20_sigmoid_ragged", 30, 5000, 20, SG, renorm=1),
    W("e8160_k36_sigmoid_bias", 40, 8160, 36, SG, renorm=1, scaling=2.5, bias_range=0.1),
    W("e8192_k8_bf16", 50, 8192, 8, SM, BF16),
]


def gpu_inputs(w, logits=None):
    x = w.make_logits() if logits is None else logits
    b = w.make_bias()
    return x, b, x.cuda(), (b.cuda() if b is not None else None)


def gpu_route(mr, w, xg, bg, path, dense=True, compact=True, status=None):
    mr.moe_router_set_topk_path(8, path)
    try:
        return mr.route(xg, w.topk, dense=dense, compact=compact, score_fn=w.score_fn, renorm=w.renorm,
                        n_group=w.n_group, topk_group=w.topk_group, n_shared=w.n_shared,
                        scaling=w.scaling, shared_weight=w.shared_weight, bias=bg, status=status)
    finally:
        mr.moe_router_set_topk_path(8, 0)


def oracle_route(orc, w, x, b, rows=None):
    xf = x.float().numpy()
    if rows is not None:
        xf = xf[rows]
    return orc.router_fwd(xf, w.topk, w.score_fn, w.renorm, w.n_group, w.topk_group, w.n_shared, w.scaling,
                          w.shared_weight, None if b is None else b.numpy())


def check_fwd(out, ref, w, rows=None, what=""):
    def sel(t):
        t = t if rows is None else t[torch.as_tensor(rows, device=t.device)]
        return t

    if "topk_idx" in out:
        assert_equal(sel(out["topk_idx"]), ref["topk_idx"], f"{what} topk_idx")
        assert_close(sel(out["topk_w"]), ref["topk_w"], f"{what} topk_w")
    if "routing_map" in out:
        assert_equal(sel(out["routing_map"]), ref["routing_map"], f"{what} routing_map")
        assert_close(sel(out["intermediate"]), ref["intermediate"], f"{what} intermediate")
        if out["probs"].dtype == torch.bfloat16:
            assert_bf16_close(sel(out["probs"]), ref["probs"], f"{what} probs(bf16)")
        else:
            assert_close(sel(out["probs"]), ref["probs"], f"{what} probs")


@pytest.mark.parametrize("compact", [True, False], ids=["compact", "dense_only"])
@pytest.mark.parametrize("path", [ARGMAX, SELECT], ids=["argmax", "select"])
@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_fwd_matches_oracle(mr, orc, w, path, compact):
    x, b, xg, bg = gpu_inputs(w)
    out = gpu_route(mr, w, xg, bg, path, compact=compact)
    torch.cuda.synchronize()
    check_fwd(out, oracle_route(orc, w, x, b), w, what=w.name)
    if w.n_group == 0 and path == ARGMAX and compact:
        note_near_ties(orc, w.name, x, w.topk - w.n_shared, w.score_fn, b)


def _tie_logits(kind, T, E):
    g = torch.Generator().manual_seed(9)
    if kind == "integers":
        return torch.randint(-3, 4, (T, E), generator=g).float()
    if kind == "all_equal":
        return torch.full((T, E), 0.5)
    if kind == "signed_zeros":
        x = torch.zeros(T, E)
        x[:, ::2] = -0.0
        x[:, ::7] = 1.0
        return x
    if kind == "saturated_sigmoid":  # every sigmoid rounds to 1.0: ties decided by index
        return 20.0 + torch.rand(T, E, generator=g)
    if kind == "two_values":
        return torch.where(torch.rand(T, E, generator=g) < 0.05, 1.0, 0.0)
    raise ValueError(kind)


@pytest.mark.parametrize("compact", [True, False], ids=["compact", "dense_only"])
@pytest.mark.parametrize("path", [ARGMAX, SELECT], ids=["argmax", "select"])
@pytest.mark.parametrize("kind", ["integers", "all_equal", "signed_zeros", "saturated_sigmoid", "two_values"])
@pytest.mark.parametrize("E,k,fn,T,dt", [(512, 36, SM, 96, F32), (256, 8, SG, 96, F32), (2304, 36, SG, 96, F32),
                                          (64, 3, SM, 96, F32), (2304, 36, SM, 3500, F32), (256, 8, SM, 96, BF16),
                                          (512, 36, SM, 96, BF16), (100, 37, SM, 50, BF16)])
def test_ties_go_to_lower_index(mr, orc, kind, E, k, fn, T, dt, path, compact):
    # T=3500 gives every CTA of the persistent softmax wide-row grid several rows;
    # dense_only takes the set-only selection (no candidate rank); bf16 softmax
    # rows take the packed arg-max rounds
    w = W(f"ties_{kind}", T, E, k, fn, dt, renorm=1)
    x = _tie_logits(kind, w.T, E)
    if dt == BF16:
        x = x.to(torch.bfloat16)
    xg = x.cuda()
    out = gpu_route(mr, w, xg, None, path, compact=compact)
    torch.cuda.synchronize()
    check_fwd(out, oracle_route(orc, w, x, None), w, what=f"{kind}")


FULL = [synth.large_softmax(k) for k in synth.LARGE_TOPKS] + [synth.large_e_softmax(), synth.large_e_sigmoid(),
                                                             synth.prefill_grouped()]


@pytest.mark.parametrize("w", FULL, ids=lambda w: w.name)
def test_full_size_sampled_rows(mr, orc, w):
    """The full workload in the benchmark's launch configuration; the oracle
    checks 2048 sampled rows one by one."""
    x, b, xg, bg = gpu_inputs(w)
    dense = w.n_group == 0
    out = gpu_route(mr, w, xg, bg, 0, dense=dense)
    torch.cuda.synchronize()
    rows = sample_rows(w.T, 2048)
    check_fwd(out, oracle_route(orc, w, x, b, rows), w, rows=rows, what=w.name)
    if w.n_group == 0:
        note_near_ties(orc, f"{w.name} (sampled rows)", x[rows], w.topk - w.n_shared, w.score_fn, b)
    # properties over every row: topk distinct, routing_map consistent with topk_idx
    idx = out["topk_idx"][:, : w.topk - w.n_shared].long()
    srt = torch.sort(idx, dim=1).values
    assert bool((srt[:, 1:] != srt[:, :-1]).all())
    if dense:
        m = torch.zeros(w.T, w.E, dtype=torch.uint8, device="cuda").scatter_(1, idx, 1)
        assert torch.equal(m, out["routing_map"])


@pytest.mark.parametrize("compact", [True, False], ids=["compact", "dense_only"])
@pytest.mark.parametrize("path", [ARGMAX, SELECT], ids=["argmax", "select"])
@pytest.mark.parametrize("E,k,fn", [(512, 36, SM), (512, 22, SG), (2304, 36, SM), (384, 8, SG)])
def test_rows_of_varying_scale_every_row(mr, orc, E, k, fn, path, compact):
    """Many rows per warp (T=8192 on the persistent grid), with per-row scales from
    1e-3 to 1e2, shifts and occasional constant rows, so the threshold a warp carries
    from one row to the next is often wrong; every row is checked."""
    T = 8192
    g = torch.Generator().manual_seed(4)
    x = torch.randn(T, E, generator=g)
    scale = 10.0 ** (torch.rand(T, 1, generator=g) * 5 - 3)
    shift = torch.randn(T, 1, generator=g) * 5
    x = x * scale + shift
    x[::97] = 0.25  # constant rows: all ties
    x = x.contiguous()
    w = W("varying", T, E, k, fn, renorm=1)
    out = gpu_route(mr, w, x.cuda(), None, path, compact=compact)
    torch.cuda.synchronize()
    check_fwd(out, oracle_route(orc, w, x, None), w, what=f"varying E={E} k={k}")
    if path == ARGMAX and compact:
        note_near_ties(orc, f"varying scale E={E} k={k} fn={fn}", x, k, fn)


BWD_CASES = [synth.tiny(), W("e512_k22", 300, 512, 22, sigma=2.0), W("e512_k22_sig", 300, 512, 22, SG),
             W("e2304_k36", 150, 2304, 36), W("e2304_k36_sig", 150, 2304, 36, SG, renorm=1, scaling=2.5,
                                                 bias_range=0.1),
             W("e100_k5_renorm", 90, 100, 5, SM, renorm=1, scaling=0.7), W("e37_sig", 40, 37, 4, SG, renorm=1),
             W("e4096_k36_wide", 60, 4096, 36), W("e8160_k36_sig_wide", 40, 8160, 36, SG, renorm=1, scaling=2.5,
                                                  bias_range=0.1),
             W("e8192_k8_renorm_wide", 40, 8192, 8, SM, renorm=1, scaling=1.5), W("e5001_sig_wide", 30, 5001, 9, SG)]


@pytest.mark.parametrize("w", BWD_CASES, ids=lambda w: w.name)
def test_bwd_matches_oracle(mr, orc, w):
    x, b, xg, bg = gpu_inputs(w)
    out = gpu_route(mr, w, xg, bg, 0, compact=False)
    g = (synth.grad(w.T, w.E).cuda() * out["routing_map"]).contiguous()
    p = mr.params_for(xg, w.topk, score_fn=w.score_fn, renorm=w.renorm, scaling=w.scaling, bias=bg)
    dx = mr.route_bwd(p, g, out["intermediate"], out["routing_map"])
    torch.cuda.synchronize()
    ref = orc.router_bwd(g.cpu().double().numpy(), out["intermediate"].cpu().double().numpy(),
                         out["routing_map"].cpu().numpy(), w.score_fn, w.renorm, w.scaling)
    assert_close(dx, ref, f"{w.name} grad_logits")


BWD_BF16_CASES = [W("e2304_k36_bf16", 150, 2304, 36, SM, BF16), W("e2304_k36_sig_bf16", 150, 2304, 36, SG, BF16,
                                                                   renorm=1, scaling=2.5, bias_range=0.1),
                  W("e512_k22_bf16", 300, 512, 22, SM, BF16, sigma=2.0),
                  W("e100_k5_renorm_bf16", 90, 100, 5, SM, BF16, renorm=1, scaling=0.7),
                  W("e37_sig_bf16", 40, 37, 4, SG, BF16, renorm=1),
                  W("e8192_k36_bf16_wide", 40, 8192, 36, SM, BF16)]


@pytest.mark.parametrize("w", BWD_BF16_CASES, ids=lambda w: w.name)
def test_bwd_bf16_grads_match_oracle(mr, orc, w):
    """bf16 logits: grad_probs in and grad_logits out in bf16, the intermediate in
    fp32; grad_logits must be a correct bf16 rounding of a value within the fp32
    bound of the oracle's gradient of the same (bf16) inputs."""
    x, b, xg, bg = gpu_inputs(w)
    out = gpu_route(mr, w, xg, bg, 0, compact=False)
    g = (synth.grad(w.T, w.E).cuda() * out["routing_map"]).to(torch.bfloat16).contiguous()
    p = mr.params_for(xg, w.topk, score_fn=w.score_fn, renorm=w.renorm, scaling=w.scaling, bias=bg)
    dx = mr.route_bwd(p, g, out["intermediate"], out["routing_map"])
    torch.cuda.synchronize()
    assert dx.dtype == torch.bfloat16
    ref = orc.router_bwd(g.cpu().double().numpy(), out["intermediate"].cpu().double().numpy(),
                         out["routing_map"].cpu().numpy(), w.score_fn, w.renorm, w.scaling)
    assert_bf16_close(dx, ref, f"{w.name} grad_logits (bf16)")


@pytest.mark.parametrize("w", [synth.large_softmax(22), synth.large_e_softmax(), synth.large_e_sigmoid()],
                         ids=lambda w: w.name)
def test_bwd_full_size_sampled_rows(mr, orc, w):
    x, b, xg, bg = gpu_inputs(w)
    out = gpu_route(mr, w, xg, bg, 0, compact=False)
    g = (synth.grad(w.T, w.E).cuda() * out["routing_map"]).contiguous()
    p = mr.params_for(xg, w.topk, score_fn=w.score_fn, renorm=w.renorm, scaling=w.scaling, bias=bg)
    dx = mr.route_bwd(p, g, out["intermediate"], out["routing_map"])
    torch.cuda.synchronize()
    rows = torch.as_tensor(sample_rows(w.T, 300), device="cuda")
    ref = orc.router_bwd(g[rows].cpu().double().numpy(), out["intermediate"][rows].cpu().double().numpy(),
                         out["routing_map"][rows].cpu().numpy(), w.score_fn, w.renorm, w.scaling)
    assert_close(dx[rows], ref, f"{w.name} grad_logits")


AUX_CASES = [W("aux_e512_k22", 300, 512, 22, sigma=2.0), W("aux_e512_k22_sig", 300, 512, 22, SG),
             W("aux_e2304_k36", 100, 2304, 36), W("aux_e2304_k36_sig", 100, 2304, 36, SG),
             W("aux_e8_k2", 16, 8, 2), W("aux_e100_k5_bf16", 80, 100, 5, SG, BF16),
             W("aux_e8160_k36", 40, 8160, 36), W("aux_e6000_k22_sig", 30, 6000, 22, SG)]


@pytest.mark.parametrize("w", AUX_CASES, ids=lambda w: w.name)
def test_aux_scores_match_oracle(mr, orc, w):
    x, _, xg, _ = gpu_inputs(w)
    out = mr.aux_scores(xg, w.topk, w.score_fn)
    g = synth.grad(w.T, w.E).cuda()
    dx = mr.aux_scores_bwd(g, out["scores"], w.score_fn)
    torch.cuda.synchronize()
    ref = orc.aux_scores_fwd(x.float().numpy(), w.topk, w.score_fn)
    assert_equal(out["routing_map"], ref["routing_map"], f"{w.name} aux routing_map")
    assert_close(out["scores"], ref["scores"], f"{w.name} aux scores")
    refdx = orc.aux_scores_bwd(g.cpu().double().numpy(), out["scores"].cpu().double().numpy(), w.score_fn)
    assert_close(dx, refdx, f"{w.name} aux grad")


def test_outputs_stay_inside_their_rows(mr):
    """Guard bands around every output: nothing is written outside [0, T*E)."""
    w = W("canary", 37, 130, 7, SG, renorm=1, bias_range=0.1)
    x, b, xg, bg = gpu_inputs(w)
    pad = 4096
    T, E, k = w.T, w.E, w.topk
    bufs = {n: torch.full((T * E + 2 * pad,), 7, dtype=d, device="cuda") for n, d in
            [("probs", torch.float32), ("routing_map", torch.uint8), ("intermediate", torch.float32)]}
    bufs["topk_idx"] = torch.full((T * k + 2 * pad,), 7, dtype=torch.int32, device="cuda")
    bufs["topk_w"] = torch.full((T * k + 2 * pad,), 7, dtype=torch.float32, device="cuda")
    views = {n: t[pad:-pad] for n, t in bufs.items()}
    p = mr.params_for(xg, k, score_fn=SG, renorm=1, bias=bg)
    mr.moe_router_fwd(p, xg, views["probs"], views["routing_map"], views["intermediate"], views["topk_idx"],
                      views["topk_w"])
    torch.cuda.synchronize()
    for n, t in bufs.items():
        assert bool((t[:pad] == 7).all()) and bool((t[-pad:] == 7).all()), n


def test_device_exp_matches_its_specification_bit_for_bit(mr, orc):
    g = torch.Generator().manual_seed(2)
    bits = torch.randint(0, 2**31 - 1, (1 << 22,), generator=g, dtype=torch.int64)
    rnd = (bits.to(torch.int32)).view(torch.float32)
    grid = torch.linspace(-110.0, 95.0, 1 << 22)
    special = torch.tensor([0.0, -0.0, 1.0, -1.0, 88.72, 88.73, 89.0, -87.3, -103.9, -104.0, -104.1,
                            float("inf"), float("-inf"), 1e-30, -1e-30, 0.34657359], dtype=torch.float32)
    x = torch.cat([rnd, -rnd, grid, special]).contiguous()
    assert x.dtype == torch.float32
    x = x[~torch.isnan(x)]
    y = torch.empty_like(x, device="cuda")
    xg = x.cuda()
    mr.moe_router_expf(xg, y)
    torch.cuda.synchronize()
    ref = orc.expf(x.numpy())
    yc = y.cpu().numpy()
    # the diagnostic writes a NaN wherever the device's packed and scalar forms
    # (exp_spec2 / exp_spec, exp_value2 / exp_value) disagree
    assert int(np.isnan(yc).sum()) == 0, "packed and scalar device exponentials disagree"
    assert np.array_equal(yc.view(np.uint32), ref.view(np.uint32))
    # and within CUDA's own expf error bound (2 ulp) of the device's expf
    cuda_exp = torch.exp(xg).cpu().numpy().astype(np.float64)
    fin = np.isfinite(cuda_exp) & (np.abs(cuda_exp) >= np.finfo(np.float32).tiny)
    ulp = np.spacing(cuda_exp[fin].astype(np.float32)).astype(np.float64)
    assert np.max(np.abs(yc[fin].astype(np.float64) - cuda_exp[fin]) / ulp) <= 2.0


def test_softmax_value_exp_error_bound(mr):
    """The exponential of the softmax numerators exp(x - max), x - max <= 0, against
    exp in double precision: relative error at most 2^-21 plus ln 2 * |x log2 e| *
    2^-24 (the one rounding of x log2 e) where the result is a normal fp32 number;
    below that it flushes towards zero (absolute error under 2^-126)."""
    gen = torch.Generator().manual_seed(11)
    x = torch.cat([torch.linspace(-104.0, 0.0, 1 << 21), -torch.rand(1 << 20, generator=gen) * 16.0,
                   -torch.rand(1 << 18, generator=gen) * 1e-3,
                   torch.tensor([0.0, -0.0, -1e-30, -0.5, -1.0, -87.0, -87.4, -88.0, -200.0, float("-inf")])])
    x = x.to(torch.float32).contiguous()
    y = torch.empty_like(x, device="cuda")
    mr.moe_router_exp_value(x.cuda(), y)
    torch.cuda.synchronize()
    xd = x.numpy().astype(np.float64)
    yd = y.cpu().numpy().astype(np.float64)
    ref = np.exp(xd)
    tiny = float(np.finfo(np.float32).tiny)
    normal = ref >= tiny
    bound = 2.0 ** -21 + np.abs(xd[normal]) * 2.0 ** -24  # ln 2 * |x log2 e| = |x|
    rel = np.abs(yd[normal] - ref[normal]) / ref[normal]
    assert np.all(rel <= bound), f"max relative error {rel.max():.3g}"
    assert np.all(np.abs(yd[~normal] - ref[~normal]) <= tiny)
    assert np.all(yd[x.numpy() == 0.0] == 1.0)


@pytest.mark.parametrize("w", [synth.large_softmax(36), synth.large_softmax(8), synth.large_e_softmax(),
                               synth.large_e_sigmoid()], ids=lambda w: w.name)
def test_aux_scores_full_size_sampled_rows(mr, orc, w):
    """The aux-scores forward at the benchmark's full sizes (its selection runs as a
    set, with no candidate rank): 2048 sampled rows against the oracle, and the
    map's row sums over every row."""
    x, _, xg, _ = gpu_inputs(w)
    out = mr.aux_scores(xg, w.topk, w.score_fn)
    torch.cuda.synchronize()
    rows = sample_rows(w.T, 2048)
    ref = orc.aux_scores_fwd(x.float().numpy()[rows], w.topk, w.score_fn)
    r = torch.as_tensor(rows, device="cuda")
    assert_equal(out["routing_map"][r], ref["routing_map"], f"{w.name} aux routing_map")
    assert_close(out["scores"][r], ref["scores"], f"{w.name} aux scores")
    assert bool((out["routing_map"].sum(dim=1, dtype=torch.int32) == w.topk).all())
