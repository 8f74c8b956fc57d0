"""Pins for the CPU oracle, against facts fixed by the pages and by mathematics.

No GPU. Each test checks the oracle against something other than itself: the
hand-derived closed forms in tests/golden, brute force over all k-subsets,
library routines on special cases (torch stable sort, softmax, sigmoid, exp),
finite differences for the backward, and invariants (weights sum to the
scaling factor under renormalisation, softmax gradients sum to zero, the sort
is a stable permutation padded to block_m).
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")
SM, SG = synth.SOFTMAX, synth.SIGMOID


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


# --------------------------------------------------------------------------- exp / sigmoid


def test_expf_sweep_within_one_ulp_of_double_exp(orc):
    x = np.linspace(-87.0, 88.0, 3_000_001, dtype=np.float64).astype(np.float32)
    y = orc.expf(x).astype(np.float64)
    ref = np.exp(x.astype(np.float64))
    ulp = np.spacing(ref.astype(np.float32)).astype(np.float64)
    assert np.max(np.abs(y - ref) / ulp) <= 1.0


def test_expf_random_bit_patterns(orc):
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 2**32, size=2_000_000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x) & (x > -103.0) & (x < 88.7)]
    y = orc.expf(x).astype(np.float64)
    ref = np.exp(x.astype(np.float64))
    normal = ref >= np.finfo(np.float32).tiny
    ulp = np.spacing(ref[normal].astype(np.float32)).astype(np.float64)
    assert np.max(np.abs(y[normal] - ref[normal]) / ulp) <= 1.0
    # subnormal results: within one subnormal step
    assert np.max(np.abs(y[~normal] - ref[~normal])) <= 2.0**-149


def test_expf_special_values_and_monotone(orc):
    y = orc.expf(np.array([0.0, -0.0, 89.0, 1000.0, -104.0, -1000.0, np.inf, -np.inf], np.float32))
    assert y[0] == 1.0 and y[1] == 1.0
    assert np.isinf(y[2]) and np.isinf(y[3]) and np.isinf(y[6])
    assert y[4] == 0.0 and y[5] == 0.0 and y[7] == 0.0
    assert np.isnan(orc.expf(np.array([np.nan], np.float32))[0])
    x = np.sort(np.random.default_rng(3).uniform(-100, 88, 500_000).astype(np.float32))
    assert np.all(np.diff(orc.expf(x)) >= 0)


def test_sigmoidf_against_double_and_symmetry(orc):
    x = np.linspace(-30, 30, 600_001).astype(np.float32)
    s = orc.sigmoidf(x).astype(np.float64)
    ref = 1.0 / (1.0 + np.exp(-x.astype(np.float64)))
    # exp (<= 2^-23 relative), the add and the divide (2^-24 each): 2^-22 in all
    assert np.max(np.abs(s - ref) / ref) <= 2.0**-22
    assert np.max(np.abs(s + orc.sigmoidf(-x) - 1.0)) <= 2.0**-23


# --------------------------------------------------------------------------- golden closed forms


@pytest.mark.parametrize("case", _golden()["cases"], ids=lambda c: c["name"])
def test_golden_router_cases(orc, case):
    fn = SM if case["score_fn"] == "softmax" else SG
    x = np.array([case["logits"]], np.float32)
    out = orc.router_fwd(x, case["topk"], fn, case.get("renorm", 0), case.get("n_group", 0),
                         case.get("topk_group", 0), case.get("n_shared", 0), case.get("scaling", 1.0),
                         case.get("shared_weight", 1.0), case.get("bias"))
    assert out["topk_idx"][0].tolist() == case["topk_idx"]
    np.testing.assert_allclose(out["topk_w"][0], case["topk_w"], rtol=1e-6, atol=1e-7)
    if "intermediate" in case:
        np.testing.assert_allclose(out["intermediate"][0], case["intermediate"], rtol=1e-6, atol=1e-7)
    if "probs" in case:
        np.testing.assert_allclose(out["probs"][0], case["probs"], rtol=1e-6, atol=1e-7)


@pytest.mark.parametrize("case", _golden()["sort_cases"], ids=lambda c: c["name"])
def test_golden_sort_cases(orc, case):
    out = orc.sort(np.array(case["topk_idx"], np.int32), np.array(case["topk_w"], np.float32),
                   case["E_tot"], case["block_m"])
    assert out["num_tokens_post_pad"] == case["num_tokens_post_pad"]
    assert out["sorted_token_ids"].tolist() == case["sorted_token_ids"]
    assert out["sorted_weights"].tolist() == case["sorted_weights"]
    assert out["expert_ids"].tolist() == case["expert_ids"]


# --------------------------------------------------------------------------- selection


def _brute_force_topk(keys: np.ndarray, k: int):
    """The unique k-subset whose every member beats every non-member
    (larger key, or equal key and lower index)."""
    E = keys.shape[0]
    found = []
    for sub in itertools.combinations(range(E), k):
        inside = set(sub)
        ok = all((keys[i] > keys[j]) or (keys[i] == keys[j] and i < j)
                 for i in inside for j in range(E) if j not in inside)
        if ok:
            found.append(sub)
    assert len(found) == 1
    return set(found[0])


@pytest.mark.parametrize("k", [1, 2, 3, 5])
@pytest.mark.parametrize("ties", [False, True])
def test_topk_set_matches_brute_force_softmax(orc, k, ties):
    rng = np.random.default_rng(11 + k)
    if ties:
        x = rng.integers(-2, 3, size=(40, 8)).astype(np.float32)  # many equal keys
    else:
        x = rng.standard_normal((40, 8)).astype(np.float32)
    out = orc.router_fwd(x, k, SM)
    for t in range(x.shape[0]):
        assert set(out["topk_idx"][t].tolist()) == _brute_force_topk(x[t], k)
        assert out["routing_map"][t].sum() == k


def test_topk_set_matches_brute_force_sigmoid_bias(orc):
    rng = np.random.default_rng(5)
    x = rng.standard_normal((40, 8)).astype(np.float32)
    b = rng.uniform(-0.1, 0.1, 8).astype(np.float32)
    out = orc.router_fwd(x, 3, SG, bias=b)
    keys = orc.sigmoidf(x) + b[None, :]  # fp32 adds, as the oracle's keys
    for t in range(x.shape[0]):
        assert set(out["topk_idx"][t].tolist()) == _brute_force_topk(keys[t], 3)


def test_topk_order_matches_torch_stable_sort(orc):
    x = synth.logits(64, 512, sigma=2.0)
    for k in (4, 8, 22, 36):
        out = orc.router_fwd(x.numpy(), k, SM)
        ref = torch.sort(x, dim=1, descending=True, stable=True).indices[:, :k]
        assert np.array_equal(out["topk_idx"], ref.numpy().astype(np.int32))
    # with ties: integer-valued logits
    xi = torch.randint(-3, 4, (64, 64), generator=torch.Generator().manual_seed(1)).float()
    out = orc.router_fwd(xi.numpy(), 10, SM)
    ref = torch.sort(xi, dim=1, descending=True, stable=True).indices[:, :10]
    assert np.array_equal(out["topk_idx"], ref.numpy().astype(np.int32))


def test_sigmoid_order_matches_torch_stable_sort_on_keys(orc):
    x = synth.logits(64, 256).numpy()
    b = synth.uniform(256, -0.1, 0.1).numpy()
    keys = torch.from_numpy(orc.sigmoidf(x) + b[None, :])
    out = orc.router_fwd(x, 9, SG, bias=b)
    ref = torch.sort(keys, dim=1, descending=True, stable=True).indices[:, :9]
    assert np.array_equal(out["topk_idx"], ref.numpy().astype(np.int32))


def test_all_equal_logits(orc):
    x = np.full((3, 16), 0.7, np.float32)
    out = orc.router_fwd(x, 5, SM, renorm=1, scaling=2.0)
    assert (out["topk_idx"] == np.arange(5)).all()
    np.testing.assert_allclose(out["topk_w"], 2.0 / 5, rtol=1e-12)
    out = orc.router_fwd(x, 5, SM, renorm=0, scaling=1.0)
    np.testing.assert_allclose(out["topk_w"], 1.0 / 16, rtol=1e-12)


# --------------------------------------------------------------------------- weights


def test_softmax_renorm_equals_softmax_over_selected_logits(orc):
    x = synth.logits(32, 64)
    out = orc.router_fwd(x.numpy(), 6, SM, renorm=1, scaling=1.7)
    idx = torch.from_numpy(out["topk_idx"]).long()
    sel = torch.gather(x.double(), 1, idx)
    ref = torch.softmax(sel, dim=1) * float(np.float32(1.7))  # the factor crosses as fp32
    np.testing.assert_allclose(out["topk_w"], ref.numpy(), rtol=1e-12)


def test_softmax_intermediate_equals_torch_softmax(orc):
    x = synth.logits(32, 300, sigma=2.0)
    out = orc.router_fwd(x.numpy(), 4, SM)
    np.testing.assert_allclose(out["intermediate"], torch.softmax(x.double(), 1).numpy(), rtol=1e-12)
    # probs = intermediate at the chosen experts, zero elsewhere (no renorm, scaling 1)
    np.testing.assert_allclose(out["probs"], out["intermediate"] * out["routing_map"], rtol=0, atol=0)


def test_sigmoid_k_equals_E_no_renorm_is_scaled_sigmoid(orc):
    x = synth.logits(16, 24)
    out = orc.router_fwd(x.numpy(), 24, SG, renorm=0, scaling=3.0)
    np.testing.assert_allclose(out["probs"], 3.0 * torch.sigmoid(x.double()).numpy(), rtol=1e-12)
    assert out["routing_map"].all()


@pytest.mark.parametrize("fn", [SM, SG])
def test_renorm_weights_sum_to_scaling(orc, fn):
    x = synth.logits(50, 128)
    out = orc.router_fwd(x.numpy(), 7, fn, renorm=1, scaling=2.827)
    c = float(np.float32(2.827))
    np.testing.assert_allclose(out["topk_w"].sum(1), c, rtol=1e-12)
    np.testing.assert_allclose(out["probs"].sum(1), c, rtol=1e-12)


def test_shared_expert_slots(orc):
    x = synth.logits(10, 40)
    out = orc.router_fwd(x.numpy(), 6, SG, renorm=1, scaling=2.0, n_shared=2, shared_weight=0.5)
    assert (out["topk_idx"][:, 4] == 40).all() and (out["topk_idx"][:, 5] == 41).all()
    assert (out["topk_w"][:, 4:] == 0.5).all()
    np.testing.assert_allclose(out["topk_w"][:, :4].sum(1), 2.0, rtol=1e-12)
    assert out["routing_map"].sum(1).tolist() == [4] * 10


# --------------------------------------------------------------------------- groups


def _group_properties(keys, sel, E, G, gk, k_r):
    gs = E // G
    m = k_r // gk
    score = []
    for g in range(G):
        top = np.sort(keys[g * gs:(g + 1) * gs])[::-1][:m]
        acc = np.float32(top[0])
        for v in top[1:]:
            acc = np.float32(acc + np.float32(v))
        score.append(acc)
    order = sorted(range(G), key=lambda g: (-score[g], g))
    kept = set(order[:gk])
    assert {e // gs for e in sel} <= kept
    pool = [e for e in range(E) if e // gs in kept]
    ref = sorted(pool, key=lambda e: (-keys[e], e))[:k_r]
    assert list(sel) == ref


def test_group_limited_selection_properties(orc):
    w = synth.Workload("g", 64, 384, 9, SG, synth.F32, renorm=1, scaling=2.827, n_group=8,
                       topk_group=4, n_shared=1, bias_range=0.05, zipf_s=1.1)
    x = w.make_logits().numpy()
    b = w.make_bias().numpy()
    out = orc.router_fwd(x, 9, SG, 1, 8, 4, 1, 2.827, 1.0, b)
    keys = orc.sigmoidf(x) + b[None, :]
    for t in range(x.shape[0]):
        _group_properties(keys[t], out["topk_idx"][t, :8], 384, 8, 4, 8)
    assert (out["topk_idx"][:, 8] == 384).all()


def test_group_limit_special_cases_reduce_to_plain_topk(orc):
    x = synth.logits(20, 48).numpy()
    plain = orc.router_fwd(x, 6, SG)["topk_idx"]
    one_group = orc.router_fwd(x, 6, SG, n_group=1, topk_group=1)["topk_idx"]
    all_groups = orc.router_fwd(x, 6, SG, n_group=48, topk_group=6)["topk_idx"]
    keep_all = orc.router_fwd(x, 6, SG, n_group=6, topk_group=6)["topk_idx"]
    assert np.array_equal(plain, one_group)
    assert np.array_equal(plain, all_groups)
    assert np.array_equal(plain, keep_all)


def test_rejected_arguments(orc):
    x = np.zeros((2, 8), np.float32)
    for kw in (dict(topk=9), dict(topk=0), dict(topk=2, n_group=3, topk_group=1),
               dict(topk=3, n_group=2, topk_group=2), dict(topk=2, n_group=2, topk_group=3),
               dict(topk=2, n_shared=2)):
        with pytest.raises(orc.OracleError):
            orc.router_fwd(x, score_fn=SG, **kw)
    with pytest.raises(orc.OracleError):
        orc.router_fwd(x, 2, SM, bias=np.zeros(8, np.float32))
    with pytest.raises(orc.OracleError):
        orc.router_fwd(x, 2, SM, n_group=2, topk_group=1)


# --------------------------------------------------------------------------- backward


def _fd_check(orc, fwd, bwd_dx, x, g, h=1e-3):
    """Central differences of L = sum(g * fwd(x)) in double, one element at a time.
    Rows whose selection flips inside [x-h, x+h] are skipped."""
    T, E = x.shape
    base_map = fwd(x)[1]
    checked = 0
    for t in range(T):
        for i in range(E):
            xp = x[t:t + 1].copy()
            xm = x[t:t + 1].copy()
            xp[0, i] = np.float32(x[t, i] + h)
            xm[0, i] = np.float32(x[t, i] - h)
            pp, mp = fwd(xp)
            pm, mm = fwd(xm)
            if not (np.array_equal(mp[0], base_map[t]) and np.array_equal(mm[0], base_map[t])):
                continue
            step = float(xp[0, i]) - float(xm[0, i])
            fd = float(np.sum(g[t] * (pp[0] - pm[0]))) / step
            assert abs(fd - bwd_dx[t, i]) <= 1e-6 + 1e-5 * abs(fd), (t, i, fd, bwd_dx[t, i])
            checked += 1
    assert checked > T * E // 2


@pytest.mark.parametrize("fn,renorm,scaling", [(SM, 1, 1.0), (SM, 0, 1.0), (SG, 1, 2.5), (SG, 0, 1.3)])
def test_router_bwd_matches_finite_differences(orc, fn, renorm, scaling):
    x = synth.logits(6, 12, sigma=1.5).numpy()
    g = synth.grad(6, 12).numpy().astype(np.float64)
    k = 3

    def fwd(xx):
        o = orc.router_fwd(xx, k, fn, renorm=renorm, scaling=scaling)
        return o["probs"], o["routing_map"]

    o = orc.router_fwd(x, k, fn, renorm=renorm, scaling=scaling)
    gm = g * o["routing_map"]
    dx = orc.router_bwd(gm, o["intermediate"], o["routing_map"], fn, renorm, scaling)
    _fd_check(orc, fwd, dx, x, gm)


def test_softmax_bwd_invariants(orc):
    x = synth.logits(64, 96).numpy()
    g = synth.grad(64, 96).numpy().astype(np.float64)
    o = orc.router_fwd(x, 8, SM, renorm=1, scaling=1.0)
    dx = orc.router_bwd(g * o["routing_map"], o["intermediate"], o["routing_map"], SM, 1, 1.0)
    # softmax is invariant to a shift of all logits, so each row's gradient sums to 0
    np.testing.assert_allclose(dx.sum(1), 0.0, atol=1e-15)
    # with renormalisation the softmax normaliser cancels: no gradient off the top-k
    np.testing.assert_allclose(dx * (1 - o["routing_map"]), 0.0, atol=1e-15)
    o2 = orc.router_fwd(x, 8, SM, renorm=0, scaling=1.0)
    dx2 = orc.router_bwd(g * o2["routing_map"], o2["intermediate"], o2["routing_map"], SM, 0, 1.0)
    np.testing.assert_allclose(dx2.sum(1), 0.0, atol=1e-15)
    assert np.abs(dx2 * (1 - o2["routing_map"])).max() > 1e-6


@pytest.mark.parametrize("fn", [SM, SG])
def test_aux_scores_fwd_and_bwd(orc, fn):
    x = synth.logits(8, 20).numpy()
    g = synth.grad(8, 20).numpy().astype(np.float64)
    o = orc.aux_scores_fwd(x, 4, fn)
    xd = torch.from_numpy(x).double()
    ref = torch.softmax(xd, 1) if fn == SM else torch.sigmoid(xd)
    np.testing.assert_allclose(o["scores"], ref.numpy(), rtol=1e-12)
    keys = x if fn == SM else orc.sigmoidf(x)
    top = torch.sort(torch.from_numpy(keys), dim=1, descending=True, stable=True).indices[:, :4]
    m = np.zeros_like(o["routing_map"])
    np.put_along_axis(m, top.numpy(), 1, 1)
    assert np.array_equal(o["routing_map"], m)
    dx = orc.aux_scores_bwd(g, o["scores"], fn)

    def fwd(xx):
        oo = orc.aux_scores_fwd(xx, 4, fn)
        return oo["scores"], np.zeros_like(oo["routing_map"])  # scores do not depend on the map

    _fd_check(orc, fwd, dx, x, g)


# --------------------------------------------------------------------------- sort


def _check_sort_layout(out, idx, w, E_tot, bm):
    T, k = idx.shape
    n = T * k
    ids = out["sorted_token_ids"]
    npp = out["num_tokens_post_pad"]
    assert npp % bm == 0 and len(ids) == npp
    flat = idx.reshape(-1)
    valid = (flat >= 0) & (flat < E_tot)
    cnt = np.bincount(flat[valid], minlength=E_tot)
    assert npp == int(sum(-(-c // bm) * bm for c in cnt))
    real = ids[ids != n]
    # every valid pair exactly once; each token appears once per valid slot
    assert sorted(real.tolist()) == np.nonzero(valid)[0].tolist()
    # stable argsort of the expert ids gives the same sequence of pairs
    order = torch.argsort(torch.from_numpy(flat[valid].astype(np.int64)), stable=True).numpy()
    assert np.array_equal(real, np.nonzero(valid)[0][order])
    # weights follow their pair; sentinels weigh 0
    sw = out["sorted_weights"]
    np.testing.assert_array_equal(sw[ids != n], w.reshape(-1)[real])
    assert (sw[ids == n] == 0).all()
    eids = out["expert_ids"]
    assert len(eids) == npp // bm and np.all(np.diff(eids) >= 0)
    # each block holds only its expert's pairs
    for b in range(npp // bm):
        blk = ids[b * bm:(b + 1) * bm]
        r = blk[blk != n]
        assert len(r) > 0 and (flat[r] == eids[b]).all()


@pytest.mark.parametrize("T,k,E_tot,bm,skew", [(16, 2, 8, 4, None), (333, 9, 385, 64, 1.1),
                                                (16, 8, 256, 32, None), (1000, 4, 37, 1, None),
                                                (50, 3, 5, 7, 2.0)])
def test_sort_layout_properties(orc, T, k, E_tot, bm, skew):
    idx, w = synth.random_topk_idx(T, k, E_tot, skew)
    out = orc.sort(idx.numpy(), w.numpy(), E_tot, bm)
    assert out["dropped"] == 0
    _check_sort_layout(out, idx.numpy(), w.numpy(), E_tot, bm)
    assert out["num_tokens_post_pad"] <= orc.sort_capacity(T, k, E_tot, bm)


def test_sort_drops_out_of_range_ids(orc):
    idx, w = synth.random_topk_idx(40, 3, 10)
    bad = idx.numpy().copy()
    bad[3, 1] = 10
    bad[7, 0] = -1
    out = orc.sort(bad, w.numpy(), 10, 4)
    assert out["dropped"] == 2
    _check_sort_layout(out, bad, w.numpy(), 10, 4)


def test_sort_capacity_is_tight(orc):
    # every expert non-empty with one pair each: worst padding
    idx = np.arange(12, dtype=np.int32).reshape(12, 1)
    out = orc.sort(idx, np.ones((12, 1), np.float32), 12, 8)
    assert out["num_tokens_post_pad"] == orc.sort_capacity(12, 1, 12, 8) == 96


# --------------------------------------------------------------------------- aux-loss scalar


def test_aux_loss_balanced_routing_gives_coeff(orc):
    # every expert receives topk*T/E of the slots: f_e = 1/E, and softmax rows
    # sum to one, so sum_e P_e = 1 and the loss is coeff whatever the probs are
    T, E, k, coeff = 96, 12, 3, 0.01
    x = synth.logits(T, E, sigma=2.0).float().numpy()
    probs = orc.aux_scores_fwd(x, k, SM)["scores"]
    counts = np.full(E, k * T // E, np.int32)
    assert orc.aux_loss_fwd(probs, counts, k, coeff, T) == pytest.approx(coeff, rel=1e-12)
    # uniform probabilities with balanced routing: the textbook minimum, coeff
    assert orc.aux_loss_fwd(np.full((T, E), 1.0 / E), counts, k, coeff, T) == pytest.approx(coeff, rel=1e-12)


def test_aux_loss_collapsed_routing_gives_coeff_times_E(orc):
    # top-1, every token sent to expert 0 with probability one: f_0 = P_0 = 1
    T, E, coeff = 50, 7, 0.3
    probs = np.zeros((T, E))
    probs[:, 0] = 1.0
    counts = np.zeros(E, np.int32)
    counts[0] = T
    assert orc.aux_loss_fwd(probs, counts, 1, coeff, T) == pytest.approx(coeff * E, rel=1e-12)


def test_aux_loss_scales_with_the_global_token_count(orc):
    # the counts and probabilities of this device's rows, normalised by N:
    # doubling N (the same rows, the rest of the tokens elsewhere) quarters it
    rng = np.random.default_rng(5)
    T, E, k = 40, 9, 2
    probs = rng.random((T, E))
    counts = rng.integers(0, 30, E).astype(np.int32)
    a = orc.aux_loss_fwd(probs, counts, k, 0.1, T)
    assert orc.aux_loss_fwd(probs, counts, k, 0.1, 2 * T) == pytest.approx(a / 4, rel=1e-12)


def test_aux_loss_bwd_matches_finite_differences(orc):
    rng = np.random.default_rng(6)
    T, E, k, coeff, N, g = 6, 5, 2, 0.05, 11, 1.7
    probs = rng.random((T, E))
    counts = rng.integers(0, 9, E).astype(np.int32)
    grad = orc.aux_loss_bwd(T, counts, k, coeff, N, g)
    h = 1e-3
    for t in range(T):
        for e in range(E):
            up, dn = probs.copy(), probs.copy()
            up[t, e] += h
            dn[t, e] -= h
            fd = (orc.aux_loss_fwd(up, counts, k, coeff, N) - orc.aux_loss_fwd(dn, counts, k, coeff, N)) / (2 * h)
            assert g * fd == pytest.approx(grad[t, e], rel=1e-8, abs=1e-14)


def test_tokens_per_expert_counts_columns(orc):
    # a map with a known column pattern: row t routes to experts t % E and (t + 3) % E
    T, E = 60, 10
    m = np.zeros((T, E), np.uint8)
    for t in range(T):
        m[t, t % E] = 1
        m[t, (t + 3) % E] = 1
    assert np.array_equal(orc.tokens_per_expert(m), np.full(E, 2 * T // E, np.int32))
    # from a real top-k map: the counts add up to T*k
    x = synth.logits(200, 33).float().numpy()
    rm = orc.aux_scores_fwd(x, 5, SM)["routing_map"]
    assert orc.tokens_per_expert(rm).sum() == 200 * 5


# --------------------------------------------------------------------------- near ties (informational)
def test_near_tie_gaps_in_fp32_ulps(orc):
    """The gap between the last key taken and the first left out, in fp32 ulps
    at the latter: an exact tie is 0; 1.0 against the next fp32 value below it
    (1 - 2^-24) is one ulp; k_r >= E leaves nothing out (-1); sigmoid keys
    0.5 + 2^-20 and 0.5 differ by 2^-20 = 16 ulps of 0.5 (2^-24 each)."""
    f = np.float32
    assert orc.near_tie_gaps(np.array([[3, 1, 1, 0.5]], f), 2)[0] == 0.0
    assert orc.near_tie_gaps(np.array([[1.0, f(1) - f(2 ** -24), -5]], f), 1)[0] == 1.0
    assert orc.near_tie_gaps(np.array([[1.0, 2.0]], f), 2)[0] == -1.0
    g = orc.near_tie_gaps(np.zeros((1, 2), f), 1, SG, np.array([0, 2 ** -20], f))
    assert g[0] == 16.0
    # order-free: a permutation of a row's logits leaves its gap unchanged
    x = np.random.default_rng(5).standard_normal((4, 64)).astype(f)
    perm = np.random.default_rng(6).permutation(64)
    assert np.array_equal(orc.near_tie_gaps(x, 9), orc.near_tie_gaps(x[:, perm], 9))
