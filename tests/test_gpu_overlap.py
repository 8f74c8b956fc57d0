"""Launch overlap (programmatic dependent launch) changes no result.

Every kernel of the library may be launched while the previous kernel in the
stream still runs, doing only its own set-up before it waits for that kernel.
A chain of dependent calls (the forward's outputs feed the backward and the
sort, the aux scores feed their backward), run eagerly and as a replayed CUDA
graph, must give bit-identical results with the overlap on and off."""
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


def _chain(mr, x, g, w, stream):
    with torch.cuda.stream(stream):
        out = mr.route(x, w.topk, renorm=1)
        dx = mr.route_bwd(mr.params_for(x, w.topk, renorm=1), g * out["routing_map"], out["intermediate"],
                          out["routing_map"])
        srt = mr.sort(out["topk_idx"], out["topk_w"], w.E, 32)
        aux = mr.aux_scores(x, w.topk)
        adx = mr.aux_scores_bwd(g, aux["scores"])
    return [out["probs"], out["routing_map"], out["intermediate"], out["topk_idx"], out["topk_w"], dx,
            srt["sorted_token_ids"], srt["sorted_weights"], srt["expert_ids"], srt["num_tokens_post_pad"],
            aux["scores"], aux["routing_map"], adx]


def _run(mr, overlap, graph):
    w = synth.Workload("overlap", 3000, 512, 8, synth.SOFTMAX, synth.F32, sigma=2.0)
    x = w.make_logits().cuda()
    g = synth.grad(w.T, w.E).cuda()
    s = torch.cuda.Stream()
    mr.moe_router_set_launch_overlap(overlap)
    try:
        if not graph:
            res = _chain(mr, x, g, w, s)
            torch.cuda.synchronize()
            return [r.clone() for r in res]
        _chain(mr, x, g, w, s)  # warm-up outside the capture
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=s):
            res = _chain(mr, x, g, w, s)
        for _ in range(3):
            gr.replay()
        torch.cuda.synchronize()
        return [r.clone() for r in res]
    finally:
        mr.moe_router_set_launch_overlap(True)


@pytest.mark.parametrize("graph", [False, True], ids=["eager", "graph"])
def test_overlap_on_and_off_give_identical_results(mr, graph):
    on = _run(mr, True, graph)
    off = _run(mr, False, graph)
    for i, (a, b) in enumerate(zip(on, off)):
        assert torch.equal(a, b), i


def test_sort_after_route_sees_the_routes_ids(mr, orc):
    """The fused call above its one-launch sizes is a forward followed by a sort
    of the forward's topk_idx. With the launch overlap the sort starts early, so
    it must not read topk_idx before the forward has written it: the buffer is
    filled with other valid ids (every pair on expert 0) before each call, and
    the sorted layout must still be the oracle's, call after call."""
    w = synth.Workload("route_then_sort", 300, 384, 9, synth.SIGMOID, synth.BF16, renorm=1, scaling=2.827,
                       n_group=8, topk_group=4, n_shared=1, bias_range=0.05, zipf_s=1.1, block_m=64)
    x, b = w.make_logits(), w.make_bias()
    r = orc.router_fwd(x.float().numpy(), w.topk, w.score_fn, w.renorm, w.n_group, w.topk_group, w.n_shared,
                       w.scaling, w.shared_weight, b.numpy())
    ref = orc.sort(r["topk_idx"], r["topk_w"].astype("float32"), w.E_tot, w.block_m)
    xg, bg = x.cuda(), b.cuda()
    p = mr.params_for(xg, w.topk, score_fn=w.score_fn, renorm=w.renorm, n_group=w.n_group,
                      topk_group=w.topk_group, n_shared=w.n_shared, scaling=w.scaling, bias=bg)
    nb = mr.moe_router_fused_workspace_bytes(p, w.block_m)
    ws = torch.empty(max(1, nb), dtype=torch.uint8, device="cuda")
    n = ref["num_tokens_post_pad"]
    for _ in range(20):
        idx = torch.zeros(w.T, w.topk, dtype=torch.int32, device="cuda")
        wt = torch.zeros(w.T, w.topk, dtype=torch.float32, device="cuda")
        bufs = mr.sort_buffers(w.T, w.topk, w.E_tot, w.block_m, "cuda")
        mr.moe_router_fused_fwd_sort(p, xg, w.block_m, idx, wt, bufs["sorted_token_ids"], bufs["sorted_weights"],
                                     bufs["expert_ids"], bufs["num_tokens_post_pad"], ws, nb)
        torch.cuda.synchronize()
        assert int(bufs["num_tokens_post_pad"].item()) == n
        assert (bufs["sorted_token_ids"][:n].cpu().numpy() == ref["sorted_token_ids"]).all()
