"""Wide rows staged in shared memory by bulk copies.

For E > 1024 with whole 128-element chunks and aligned rows, each warp's next
row is copied into its shared key buffer while it writes the current row's
outputs, and the copy is waited for with a bounded wait. These cases give every
warp several rows (T larger than the persistent grid's warps), in fp32 and bf16
(whose raw row sits in the buffer's upper half and is turned into keys in
place), with and without the intermediate output, and check every row against
the oracle. Afterwards the library's device status word must still be clear.

The bounded wait itself is exercised without any GPU fault: a host-side test
hook makes the kernel arm each row's barrier for the row's bytes but issue no
copy, with a wait limit of a few microseconds, so every wait runs out while no
copy is in flight. The call must report MR_ETIMEOUT in its status word (or in
the library's device word when it has none) and return, and the next normal
call must be correct.
"""
import pytest
import torch

import synth
from test_gpu_router import ARGMAX, SELECT, SG, SM, BF16, F32, W, check_fwd, gpu_inputs, gpu_route, oracle_route

pytestmark = pytest.mark.gpu

STAGED = [
    W("staged_e2304_k36_bf16_softmax", 6500, 2304, 36, SM, BF16),
    W("staged_e2304_k36_bf16_sigmoid_bias", 6500, 2304, 36, SG, BF16, renorm=1, scaling=2.5, bias_range=0.1),
    W("staged_e1536_k100_f32_sigmoid", 6500, 1536, 100, SG, F32, renorm=1),
    W("staged_e2304_k8_f32_softmax", 6500, 2304, 8, SM, F32),
    W("staged_e8192_k36_f32_softmax", 3000, 8192, 36, SM, F32),
    W("staged_e8064_k22_bf16_sigmoid", 3000, 8064, 22, SG, BF16, renorm=1, bias_range=0.1),
]


@pytest.mark.parametrize("dense", [True, False], ids=["dense", "compact_only"])
@pytest.mark.parametrize("path", [ARGMAX, SELECT], ids=["argmax", "select"])
@pytest.mark.parametrize("w", STAGED, ids=lambda w: w.name)
def test_staged_rows_every_row(mr, orc, w, path, dense):
    x, b, xg, bg = gpu_inputs(w)
    out = gpu_route(mr, w, xg, bg, path, dense=dense)
    torch.cuda.synchronize()
    check_fwd(out, oracle_route(orc, w, x, b), w, what=w.name)


def test_device_status_is_clear_after_staged_rows(mr):
    w = STAGED[0]
    _, _, xg, bg = gpu_inputs(w)
    assert mr.device_status(clear=True) == 0
    for path in (ARGMAX, SELECT):
        gpu_route(mr, w, xg, bg, path)
    out = mr.aux_scores(xg, w.topk, w.score_fn)
    torch.cuda.synchronize()
    assert out["scores"].shape == (w.T, w.E)
    assert mr.device_status() == 0


@pytest.mark.parametrize("path", [ARGMAX, SELECT], ids=["argmax", "select"])
@pytest.mark.parametrize("in_dtype", [F32, BF16], ids=["f32", "bf16"])
def test_staged_softmax_rows_far_from_the_previous_max(mr, orc, path, in_dtype):
    """Staged softmax rows shifted by offsets from -500 to +1000 in a random
    order (bf16: coarse values, many ties at the threshold), so the threshold
    and the row max a warp meets change by large steps from row to row; every
    row is checked."""
    T, E, k = 6500, 2304, 36
    g = torch.Generator().manual_seed(21)
    x = torch.randn(T, E, generator=g)
    offs = torch.tensor([0.0, 20.0, 63.0, 66.0, -70.0, 200.0, -500.0, 1000.0])
    x = x + offs[torch.randint(0, len(offs), (T, 1), generator=g)]
    if in_dtype == BF16:
        x = x.to(torch.bfloat16)
    x = x.contiguous()
    w = W("far_max", T, E, k, SM, in_dtype)
    out = gpu_route(mr, w, x.cuda(), None, path)
    torch.cuda.synchronize()
    check_fwd(out, oracle_route(orc, w, x, None), w, what="far from the previous max")


@pytest.mark.parametrize("path", [ARGMAX, SELECT], ids=["argmax", "select"])
@pytest.mark.parametrize("in_dtype", [F32, BF16], ids=["f32", "bf16"])
def test_bounded_wait_gives_up_and_reports_it(mr, orc, path, in_dtype):
    w = W("timeout", 3000, 2304, 36, SM, in_dtype)
    x, b, xg, bg = gpu_inputs(w)
    assert mr.device_status(clear=True) == 0
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mr.moe_router_set_wait_test(8, 1)
    try:
        gpu_route(mr, w, xg, bg, path, status=status)
        torch.cuda.synchronize()
        got_call = int(status.item())
        # no status word of its own: the timeout goes to the library's device word
        mr.aux_scores(xg, w.topk, w.score_fn)
        torch.cuda.synchronize()
    finally:
        mr.moe_router_set_wait_test(0, 0)
    assert got_call == mr.MR_ETIMEOUT
    assert mr.device_status(clear=True) == mr.MR_ETIMEOUT
    assert mr.device_status() == 0
    # the context is still usable and the next normal call is correct
    status.zero_()
    out = gpu_route(mr, w, xg, bg, path, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    check_fwd(out, oracle_route(orc, w, x, b), w, what="after a timeout")
    assert mr.device_status() == 0
