"""Wide rows staged in shared memory by bulk copies.

For E > 1024 with whole 128-element chunks and aligned rows, each warp's next
row is copied into its shared key buffer while it writes the current row's
outputs, and the copy is waited for with a bounded wait. These cases give every
warp several rows (T larger than the persistent grid's warps), in fp32 and bf16
(whose raw row sits in the buffer's upper half and is turned into keys in
place), with and without the intermediate output, and check every row against
the oracle. Afterwards the library's device status word must still be clear.
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
