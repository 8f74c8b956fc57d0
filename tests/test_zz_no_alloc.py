"""moe_sort_noalloc, the sort for callers that cannot allocate device memory.

Some callers are handed only a stream and their tensors (an inference-engine
plugin or a custom op without an allocator handle), or must not call cudaMalloc
because it would synchronise the device at that point. moe_sort_noalloc serves
them: it takes no workspace and keeps its scratch in a fixed device array inside
the library. These tests call it through the C ABI and check that two calls in a
row give exactly what moe_sort gives with its own workspace (the sorted layout
is compared bit for bit, as in the other sort tests), and that a problem whose
scratch would not fit the array is refused before anything runs.

This file is collected last on purpose (tests/test_zz_*), so that a run that
stops at the first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

import synth
from parity import assert_equal

pytestmark = pytest.mark.gpu


def _noalloc(mr, idx, w, E_tot, bm):
    T, k = idx.shape
    out = mr.sort_buffers(T, k, E_tot, bm, idx.device)
    status = torch.zeros(1, dtype=torch.int32, device=idx.device)
    mr.moe_sort_noalloc(idx, w, T, k, E_tot, bm, out["sorted_token_ids"], out["sorted_weights"],
                        out["expert_ids"], out["num_tokens_post_pad"], status)
    return out, status


def _check_same(ref, out, bm, what):
    n = int(ref["num_tokens_post_pad"].item())
    assert int(out["num_tokens_post_pad"].item()) == n, what
    assert_equal(out["sorted_token_ids"][:n], ref["sorted_token_ids"][:n].cpu().numpy(), f"{what} ids")
    assert_equal(out["sorted_weights"][:n].view(torch.int32), ref["sorted_weights"][:n].view(torch.int32).cpu().numpy(),
                 f"{what} weights (bits)")
    assert_equal(out["expert_ids"][: n // bm], ref["expert_ids"][: n // bm].cpu().numpy(), f"{what} expert_ids")


def test_two_calls_in_a_row_match_moe_sort(mr):
    # first a large skewed prefill-shaped sort, then a smaller one with other sizes:
    # whatever the first call left in the shared scratch must not leak into the second
    calls = [(16384, 9, 385, 64, 1.1), (1000, 4, 37, 8, None)]
    for T, k, E_tot, bm, skew in calls:
        idx, w = synth.random_topk_idx(T, k, E_tot, skew)
        idx, w = idx.cuda(), w.cuda()
        ref = mr.sort(idx, w, E_tot, bm)
        out, status = _noalloc(mr, idx, w, E_tot, bm)
        torch.cuda.synchronize()
        _check_same(ref, out, bm, f"T={T} k={k} E_tot={E_tot} block_m={bm}")
        assert int(status.item()) == 0


def test_scratch_limit_is_enforced(mr):
    # the scratch the sort needs grows with the number of 4096-pair chunks; find the
    # largest T (in whole chunks) whose scratch fits the array, with 4096 experts
    k, E_tot, bm = 1, 4096, 16
    limit = mr.moe_sort_noalloc_scratch_bytes()
    T2 = 4096
    while mr.moe_sort_workspace_bytes(T2 + 4096, k, E_tot, bm) <= limit:
        T2 += 4096
    T = T2 + 4096  # one chunk more: just over the array
    assert mr.moe_sort_workspace_bytes(T, k, E_tot, bm) > limit
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    with pytest.raises(mr.MoERouterError) as e:
        mr.moe_sort_noalloc(dummy, None, T, k, E_tot, bm, dummy, None, dummy, dummy)
    assert e.value.code == mr.MR_EUNSUPPORTED
    # the largest table that fits is accepted
    assert mr.moe_sort_workspace_bytes(T2, k, E_tot, bm) <= limit
    idx = torch.randint(0, E_tot, (T2, k), dtype=torch.int32, device="cuda")
    out, status = _noalloc(mr, idx, None, E_tot, bm)
    ref = mr.sort(idx, None, E_tot, bm)
    torch.cuda.synchronize()
    n = int(ref["num_tokens_post_pad"].item())
    assert int(out["num_tokens_post_pad"].item()) == n
    assert torch.equal(out["sorted_token_ids"][:n], ref["sorted_token_ids"][:n])
    assert np.array_equal(out["expert_ids"][: n // bm].cpu().numpy(), ref["expert_ids"][: n // bm].cpu().numpy())
