"""GPU parity of the sort and of the fused decode route+sort against the CPU
oracle, through the C ABI: the sorted layout must match exactly."""
import numpy as np
import pytest
import torch

import synth
from parity import assert_close, assert_equal

pytestmark = pytest.mark.gpu


# One CTA up to 4096 pairs; then one thread-block cluster (16 CTAs x 1024 threads
# x 2 pairs = 32768 pairs, or half that where the GPU allows clusters of 8 only;
# both sides of both limits are here); above that chunks of 1024..4096 pairs in
# clusters of 8 (a partial last cluster, fewer experts than a cluster has CTAs,
# 4096 experts over many chunks, about a million pairs).
SORT_CASES = [(16, 2, 8, 4, None), (16384, 9, 385, 64, 1.1), (16, 8, 256, 32, None), (1000, 4, 37, 1, None),
              (50, 3, 5, 7, 2.0), (4097, 6, 128, 16, None), (3, 1, 4096, 8, None), (8192, 36, 2304, 64, 0.8),
              (1, 1, 1, 1, None), (5000, 2, 3, 128, None), (1025, 4, 100, 16, None), (4096, 1, 64, 8, None),
              (20000, 3, 5, 3, None), (50000, 8, 4096, 32, 1.1), (131072, 8, 256, 32, 1.1),
              (70001, 9, 385, 64, 1.1), (2048, 16, 64, 8, None), (2049, 16, 64, 8, None),
              (1024, 16, 300, 16, 1.1), (1025, 16, 300, 16, None), (1500, 16, 2304, 32, 0.8),
              (12000, 16, 2304, 32, 0.8)]


@pytest.mark.parametrize("T,k,E_tot,bm,skew", SORT_CASES)
def test_sort_matches_oracle(mr, orc, T, k, E_tot, bm, skew):
    idx, w = synth.random_topk_idx(T, k, E_tot, skew)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = mr.sort(idx.cuda(), w.cuda(), E_tot, bm, status=status)
    torch.cuda.synchronize()
    ref = orc.sort(idx.numpy(), w.numpy(), E_tot, bm)
    n = int(out["num_tokens_post_pad"].item())
    assert n == ref["num_tokens_post_pad"]
    assert_equal(out["sorted_token_ids"][:n], ref["sorted_token_ids"], "sorted_token_ids")
    assert_equal(out["sorted_weights"][:n].view(torch.int32), ref["sorted_weights"].view(np.int32),
                 "sorted_weights (bits)")
    assert_equal(out["expert_ids"][: n // bm], ref["expert_ids"], "expert_ids")
    assert int(status.item()) == 0


def test_sort_drops_out_of_range_ids_and_flags_them(mr, orc):
    idx, w = synth.random_topk_idx(3000, 4, 40)
    bad = idx.clone()
    bad[5, 1] = 40
    bad[77, 0] = -3
    bad[2999, 3] = 1 << 30
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = mr.sort(bad.cuda(), w.cuda(), 40, 8, status=status)
    torch.cuda.synchronize()
    ref = orc.sort(bad.numpy(), w.numpy(), 40, 8)
    assert ref["dropped"] == 3
    n = int(out["num_tokens_post_pad"].item())
    assert n == ref["num_tokens_post_pad"]
    assert_equal(out["sorted_token_ids"][:n], ref["sorted_token_ids"], "sorted_token_ids")
    assert int(status.item()) == mr.MR_ERANGE


def test_sort_leaves_tails_and_guard_bands_untouched(mr):
    T, k, E_tot, bm = 700, 3, 50, 16
    idx, w = synth.random_topk_idx(T, k, E_tot)
    cap = mr.moe_sort_capacity(T, k, E_tot, bm)
    pad = 1024
    ids = torch.full((cap + 2 * pad,), -7, dtype=torch.int32, device="cuda")
    sw = torch.full((cap + 2 * pad,), -7.0, dtype=torch.float32, device="cuda")
    eids = torch.full((cap // bm + 1 + 2 * pad,), -7, dtype=torch.int32, device="cuda")
    npp = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(mr.moe_sort_workspace_bytes(T, k, E_tot, bm), dtype=torch.uint8, device="cuda")
    mr.moe_sort(idx.cuda(), w.cuda(), T, k, E_tot, bm, ids[pad:-pad], sw[pad:-pad], eids[pad:-pad], npp, ws)
    torch.cuda.synchronize()
    n = int(npp.item())
    assert bool((ids[:pad] == -7).all()) and bool((ids[pad + n:] == -7).all())
    assert bool((sw[:pad] == -7).all()) and bool((sw[pad + n:] == -7).all())
    assert bool((eids[:pad] == -7).all()) and bool((eids[pad + n // bm:] == -7).all())


def test_sort_zero_tokens(mr):
    npp = torch.full((1,), 99, dtype=torch.int32, device="cuda")
    buf = torch.empty(16, dtype=torch.int32, device="cuda")
    ws = torch.empty(1024, dtype=torch.uint8, device="cuda")
    mr.moe_sort(None, None, 0, 4, 8, 4, buf, None, buf, npp, ws)
    torch.cuda.synchronize()
    assert int(npp.item()) == 0


def _oracle_fused(orc, w, x, b):
    r = orc.router_fwd(x.float().numpy(), w.topk, w.score_fn, w.renorm, w.n_group, w.topk_group, w.n_shared,
                       w.scaling, w.shared_weight, None if b is None else b.numpy())
    s = orc.sort(r["topk_idx"], r["topk_w"].astype(np.float32), w.E_tot, w.block_m)
    return r, s


# the decode shapes exactly as benchmarked: DeepSeek-R1 (E=256, topk=8) and GPT-OSS
# (E=128, topk=4), both with block_m=32
FUSED = [synth.decode(T) for T in synth.DECODE_TS] + [synth.decode_gpt_oss(T) for T in (1, 4, 16, 32, 64)] + [
    synth.Workload("decode_T16_grouped_shared", 16, 384, 9, synth.SIGMOID, synth.BF16, renorm=1, scaling=2.827,
                   n_group=8, topk_group=4, n_shared=1, bias_range=0.05, zipf_s=1.1, block_m=64),
    synth.Workload("decode_T5_e128_k4", 5, 128, 4, synth.SOFTMAX, synth.BF16, renorm=1, block_m=16),
    # at most 32 pairs: a warp per token, one warp sorts (edges of that form)
    synth.Workload("tiny_T1_e1024_k32", 1, 1024, 32, synth.SOFTMAX, synth.F32, renorm=1, block_m=16),
    synth.Workload("tiny_T2_grouped_shared_bm24", 2, 384, 9, synth.SIGMOID, synth.BF16, renorm=1, scaling=2.827,
                   n_group=8, topk_group=4, n_shared=1, bias_range=0.05, block_m=24),
    synth.Workload("tiny_T16_e64_k2_bm1", 16, 64, 2, synth.SOFTMAX, synth.F32, renorm=1, block_m=1),
    synth.Workload("tiny_T7_e256_k4_bm3", 7, 256, 4, synth.SOFTMAX, synth.BF16, renorm=1, block_m=3),
    synth.Workload("tiny_T3_e37_k10_sigmoid", 3, 37, 10, synth.SIGMOID, synth.F32, renorm=1, scaling=1.5,
                   bias_range=0.1, block_m=8),
    synth.Workload("above_tiny_T3_e100_k11", 3, 100, 11, synth.SIGMOID, synth.F32, renorm=1, scaling=1.5,
                   bias_range=0.1, block_m=8),
    # at most 128 pairs and 16 tokens: a warp per token, one warp ranks in four slots
    synth.Workload("small_T1_e1024_k100", 1, 1024, 100, synth.SOFTMAX, synth.F32, renorm=1, block_m=16),
    synth.Workload("small_T9_e256_k8_bm24", 9, 256, 8, synth.SOFTMAX, synth.BF16, renorm=1, block_m=24),
    synth.Workload("small_T7_grouped_shared_bm48", 7, 384, 9, synth.SIGMOID, synth.BF16, renorm=1, scaling=2.827,
                   n_group=8, topk_group=4, n_shared=1, bias_range=0.05, zipf_s=1.1, block_m=48),
    synth.Workload("small_T16_e64_k8_bm1", 16, 64, 8, synth.SOFTMAX, synth.F32, renorm=1, block_m=1),
    synth.Workload("small_T11_e100_k6_sigmoid", 11, 100, 6, synth.SIGMOID, synth.F32, renorm=1, scaling=1.5,
                   bias_range=0.1, block_m=8),
    synth.Workload("above_small_T16_e128_k9", 16, 128, 9, synth.SOFTMAX, synth.BF16, renorm=1, block_m=16),
    synth.Workload("fused32_T17", 17, 256, 8, synth.SOFTMAX, synth.BF16, renorm=1, block_m=32),
    synth.Workload("fused32_T32_e256_k8", 32, 256, 8, synth.SOFTMAX, synth.BF16, renorm=1, block_m=32),
    synth.Workload("fused32_T24_e128_k4", 24, 128, 4, synth.SOFTMAX, synth.BF16, renorm=1, block_m=16),
    synth.Workload("fused32_T29_e100_sigmoid", 29, 100, 6, synth.SIGMOID, synth.F32, renorm=1, scaling=1.5,
                   bias_range=0.1, block_m=8),
    synth.Workload("fused64_T33", 33, 256, 8, synth.SOFTMAX, synth.BF16, renorm=1, block_m=32),
    synth.Workload("fused64_T64_e256_k8", 64, 256, 8, synth.SOFTMAX, synth.BF16, renorm=1, block_m=32),
    synth.Workload("fused64_T50_e128_k4_grouped", 50, 128, 4, synth.SIGMOID, synth.BF16, renorm=1, n_group=4,
                   topk_group=2, bias_range=0.05, block_m=16),
    synth.Workload("fallback_T65", 65, 256, 8, synth.SOFTMAX, synth.BF16, renorm=1, block_m=32),
    synth.Workload("fallback_T17_e384", 17, 384, 8, synth.SOFTMAX, synth.BF16, renorm=1, block_m=32),
    synth.Workload("fallback_T300_grouped", 300, 384, 9, synth.SIGMOID, synth.BF16, renorm=1, scaling=2.827,
                   n_group=8, topk_group=4, n_shared=1, bias_range=0.05, block_m=64),
    synth.Workload("fallback_wide_T4_e2304", 4, 2304, 36, synth.SOFTMAX, synth.F32, block_m=8),
    # one thread-block cluster, a warp per token, up to 512 tokens
    synth.Workload("cluster_T128_e256_k8", 128, 256, 8, synth.SOFTMAX, synth.BF16, renorm=1, block_m=32),
    synth.Workload("cluster_T512_e256_k8", 512, 256, 8, synth.SOFTMAX, synth.BF16, renorm=1, block_m=32),
    synth.Workload("cluster_T256_e128_k4", 256, 128, 4, synth.SOFTMAX, synth.BF16, renorm=1, block_m=32),
    synth.Workload("cluster_T100_e1024_k36", 100, 1024, 36, synth.SOFTMAX, synth.F32, block_m=16),
    synth.Workload("cluster_T333_e100_sigmoid", 333, 100, 6, synth.SIGMOID, synth.F32, renorm=1, scaling=1.5,
                   bias_range=0.1, block_m=8),
    synth.Workload("separate_T513_e256_k8", 513, 256, 8, synth.SOFTMAX, synth.BF16, renorm=1, block_m=32),
    # above 4096 pairs: the forward, then the one-cluster sort (or the chunked one)
    synth.Workload("prefill_T600_e256_k8", 600, 256, 8, synth.SOFTMAX, synth.BF16, renorm=1, block_m=32),
    synth.Workload("prefill_T5000_e100_k5_sigmoid", 5000, 100, 5, synth.SIGMOID, synth.F32, renorm=1, scaling=1.5,
                   bias_range=0.1, block_m=8),
    synth.Workload("prefill_T3000_grouped_shared", 3000, 384, 9, synth.SIGMOID, synth.BF16, renorm=1, scaling=2.827,
                   n_group=8, topk_group=4, n_shared=1, bias_range=0.05, zipf_s=1.1, block_m=64),
    synth.Workload("prefill_T2500_e1024_k36", 2500, 1024, 36, synth.SOFTMAX, synth.F32, block_m=16),
    synth.Workload("prefill_T9000_e64_k2", 9000, 64, 2, synth.SOFTMAX, synth.F32, renorm=1, block_m=128),
    # wide rows: the forward, then moe_sort
    synth.Workload("prefill_wide_T300_e2304", 300, 2304, 36, synth.SIGMOID, synth.F32, renorm=1, scaling=2.5,
                   bias_range=0.1, block_m=32),
]


@pytest.mark.parametrize("path", [1, 2], ids=["argmax", "select"])
@pytest.mark.parametrize("w", FUSED, ids=lambda w: w.name)
def test_fused_route_sort_matches_oracle(mr, orc, w, path):
    x = w.make_logits()
    b = w.make_bias()
    xg = x.cuda()
    bg = b.cuda() if b is not None else None
    mr.moe_router_set_topk_path(8, path)
    try:
        out = mr.fused_route_sort(xg, w.topk, w.block_m, score_fn=w.score_fn, renorm=w.renorm, n_group=w.n_group,
                                  topk_group=w.topk_group, n_shared=w.n_shared, scaling=w.scaling,
                                  shared_weight=w.shared_weight, bias=bg)
        unf = mr.route(xg, w.topk, dense=False, score_fn=w.score_fn, renorm=w.renorm, n_group=w.n_group,
                       topk_group=w.topk_group, n_shared=w.n_shared, scaling=w.scaling,
                       shared_weight=w.shared_weight, bias=bg)
        uns = mr.sort(unf["topk_idx"], unf["topk_w"], w.E_tot, w.block_m)
    finally:
        mr.moe_router_set_topk_path(8, 0)
    torch.cuda.synchronize()
    r, s = _oracle_fused(orc, w, x, b)
    assert_equal(out["topk_idx"], r["topk_idx"], "topk_idx")
    assert_close(out["topk_w"], r["topk_w"], "topk_w")
    n = int(out["num_tokens_post_pad"].item())
    assert n == s["num_tokens_post_pad"]
    assert_equal(out["sorted_token_ids"][:n], s["sorted_token_ids"], "sorted_token_ids")
    assert_equal(out["expert_ids"][: n // w.block_m], s["expert_ids"], "expert_ids")
    # weights: the fused call's sorted weights are exactly the unfused path's
    assert int(uns["num_tokens_post_pad"].item()) == n
    assert torch.equal(out["sorted_token_ids"][:n], uns["sorted_token_ids"][:n])
    assert torch.equal(out["sorted_weights"][:n], uns["sorted_weights"][:n])
    assert torch.equal(out["topk_w"], unf["topk_w"])
    ids = s["sorted_token_ids"]
    real = ids < w.T * w.topk
    refw = np.zeros(len(ids))
    refw[real] = r["topk_w"].reshape(-1)[ids[real]]
    assert_close(out["sorted_weights"][:n], refw, "sorted_weights")


@pytest.mark.parametrize("path", [0, 1, 2], ids=["auto", "argmax", "select"])
def test_fused_prefill_full_size_every_row(mr, orc, path):
    """The prefill workload (T=16384, E=384 + 1 shared, topk=9, grouped sigmoid,
    block_m=64) through moe_router_fused_fwd_sort (the forward, then the sort in
    one launch of one thread-block cluster): every row's top-k and the whole
    sorted layout against the oracle."""
    w = synth.prefill_grouped()
    x = w.make_logits()
    b = w.make_bias()
    xg, bg = x.cuda(), b.cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mr.moe_router_set_topk_path(8, path)
    try:
        out = mr.fused_route_sort(xg, w.topk, w.block_m, score_fn=w.score_fn, renorm=w.renorm, n_group=w.n_group,
                                  topk_group=w.topk_group, n_shared=w.n_shared, scaling=w.scaling,
                                  shared_weight=w.shared_weight, bias=bg, status=status)
    finally:
        mr.moe_router_set_topk_path(8, 0)
    torch.cuda.synchronize()
    r, srt = _oracle_fused(orc, w, x, b)
    assert int(status.item()) == 0
    assert_equal(out["topk_idx"], r["topk_idx"], "topk_idx")
    assert_close(out["topk_w"], r["topk_w"], "topk_w")
    n = int(out["num_tokens_post_pad"].item())
    assert n == srt["num_tokens_post_pad"]
    assert_equal(out["sorted_token_ids"][:n], srt["sorted_token_ids"], "sorted_token_ids")
    assert_equal(out["expert_ids"][: n // w.block_m], srt["expert_ids"], "expert_ids")
    # the sorted weights are the GPU's own topk_w gathered by sorted id (bit for bit)
    ids = out["sorted_token_ids"][:n].long()
    real = ids < w.T * w.topk
    want = torch.zeros(n, dtype=torch.float32, device="cuda")
    want[real] = out["topk_w"].reshape(-1)[ids[real]]
    assert torch.equal(out["sorted_weights"][:n], want)
