"""GPU parity of the aux-loss scalar (forward and backward) and of the per-expert
token counts against the CPU oracle, through the C ABI.

Inputs are seeded and made on the host: probabilities are uniform random rows
(any non-negative matrix is a valid input to the loss) and routing maps are
random 0/1 matrices, or, in the chained case, the oracle's own aux scores and
routing map of synthetic logits. The counts must match exactly; the loss and
its gradient within the fp32 tolerance of the other parity tests.
"""
import numpy as np
import pytest
import torch

import synth
from parity import assert_close, assert_equal, sample_rows

pytestmark = pytest.mark.gpu

SM = synth.SOFTMAX


def _probs(T, E, seed=11):
    g = torch.Generator().manual_seed(seed)
    return torch.rand(T, E, generator=g, dtype=torch.float32)


def _map(T, E, p, seed=12):
    g = torch.Generator().manual_seed(seed)
    return (torch.rand(T, E, generator=g) < p).to(torch.uint8)


def _loss_close(gpu, ref, what):
    assert_close(np.array([float(gpu)]), np.array([ref]), what)


CASES = [(16, 8, 2, 0.01), (1000, 64, 4, 1e-3), (300, 37, 3, 0.5), (4097, 130, 7, 0.02), (2048, 2304, 36, 1e-2)]


@pytest.mark.parametrize("T,E,k,coeff", CASES, ids=lambda v: str(v))
def test_aux_loss_and_counts_match_oracle(mr, orc, T, E, k, coeff):
    probs = _probs(T, E)
    rmap = _map(T, E, min(0.9, k / E))
    counts = mr.tokens_per_expert(rmap.cuda())
    ref_counts = orc.tokens_per_expert(rmap.numpy())
    N = T + 17  # counts and probabilities taken over more tokens than these rows
    loss = mr.aux_loss(probs.cuda(), counts, k, coeff, N)
    gl = torch.tensor([1.7], dtype=torch.float32, device="cuda")
    grad = mr.aux_loss_bwd(gl, counts, T, k, coeff, N)
    torch.cuda.synchronize()
    assert_equal(counts, ref_counts, "tokens_per_expert")
    ref = orc.aux_loss_fwd(probs.double().numpy(), ref_counts, k, coeff, N)
    _loss_close(loss.item(), ref, f"loss T={T} E={E}")
    assert_close(grad, orc.aux_loss_bwd(T, ref_counts, k, coeff, N, 1.7), f"grad_probs T={T} E={E}")


@pytest.mark.parametrize("T,E", [(70001, 16), (5000, 80), (3, 2304), (1030, 4096)], ids=lambda v: str(v))
def test_counts_of_any_nonzero_byte(mr, orc, T, E):
    """Token counts count every nonzero map byte once (values 1..255), over 64-column
    slabs with a partial last slab, chunks of rows whose counts need more than 16
    bits in all (T above 65535), and a handful of rows."""
    g = torch.Generator().manual_seed(13)
    vals = torch.randint(1, 256, (T, E), generator=g, dtype=torch.int32).to(torch.uint8)
    keep = torch.rand(T, E, generator=g) < 0.3
    rmap = torch.where(keep, vals, torch.zeros_like(vals)).contiguous()
    counts = mr.tokens_per_expert(rmap.cuda())
    torch.cuda.synchronize()
    assert_equal(counts, orc.tokens_per_expert(rmap.numpy()), f"tokens_per_expert T={T} E={E}")


def test_misaligned_rows_take_the_scalar_path(mr, orc):
    T, E, k = 500, 64, 4
    base = _probs(T * E + 1, 1).reshape(-1)
    probs = base[1:].reshape(T, E)  # 4-byte offset: no 16-byte vectors
    rmap = _map(T, E, 0.1)
    counts = torch.as_tensor(orc.tokens_per_expert(rmap.numpy())).cuda()
    pg = base.cuda()[1:].view(T, E)
    loss = mr.aux_loss(pg, counts, k, 0.1)
    gbuf = torch.zeros(T * E + 1, dtype=torch.float32, device="cuda")
    gl = torch.tensor([0.5], dtype=torch.float32, device="cuda")
    mr.moe_aux_loss_bwd(T, E, k, 0.1, T, counts, gl, gbuf[1:])
    torch.cuda.synchronize()
    _loss_close(loss.item(), orc.aux_loss_fwd(probs.double().numpy(), counts.cpu().numpy(), k, 0.1, T), "loss")
    assert_close(gbuf[1:].view(T, E), orc.aux_loss_bwd(T, counts.cpu().numpy(), k, 0.1, T, 0.5), "grad")
    assert float(gbuf[0]) == 0.0


def test_zero_tokens(mr):
    E = 16
    counts = torch.full((E,), 5, dtype=torch.int32, device="cuda")
    mr.moe_tokens_per_expert(0, E, None, counts)
    loss = torch.full((1,), 3.0, dtype=torch.float32, device="cuda")
    mr.moe_aux_loss_fwd(0, E, 2, 0.1, 1, None, counts, loss, None, 0)
    torch.cuda.synchronize()
    assert int(counts.abs().sum()) == 0 and float(loss) == 0.0


def test_chained_from_logits_at_full_size(mr, orc):
    """The aux scores and map of the headline workload's logits (oracle-computed,
    fed to both sides as fp32 scores and a uint8 map), counted and reduced on the
    GPU, against the oracle's chain."""
    w = synth.large_e_softmax()
    x = w.make_logits()
    ref = orc.aux_scores_fwd(x.float().numpy(), w.topk, SM)
    scores = torch.from_numpy(ref["scores"].astype(np.float32))
    counts = mr.tokens_per_expert(torch.from_numpy(ref["routing_map"]).cuda())
    loss = mr.aux_loss(scores.cuda(), counts, w.topk, 1e-2)
    gl = torch.tensor([1.0], dtype=torch.float32, device="cuda")
    grad = mr.aux_loss_bwd(gl, counts, w.T, w.topk, 1e-2)
    torch.cuda.synchronize()
    ref_counts = orc.tokens_per_expert(ref["routing_map"])
    assert_equal(counts, ref_counts, "tokens_per_expert")
    assert int(ref_counts.sum()) == w.T * w.topk
    _loss_close(loss.item(), orc.aux_loss_fwd(scores.double().numpy(), ref_counts, w.topk, 1e-2, w.T), "loss")
    rows = sample_rows(w.T, 64)
    g_ref = orc.aux_loss_bwd(len(rows), ref_counts, w.topk, 1e-2, w.T, 1.0)
    assert_close(grad[torch.as_tensor(rows, device="cuda")], g_ref, "grad_probs (sampled rows)")


def test_repeated_calls_are_bit_identical(mr):
    T, E, k = 8192, 2304, 36
    probs = _probs(T, E).cuda()
    counts = mr.tokens_per_expert(_map(T, E, k / E).cuda())
    a = mr.aux_loss(probs, counts, k, 0.01)
    b = mr.aux_loss(probs, counts, k, 0.01)
    torch.cuda.synchronize()
    assert a.view(torch.int32).item() == b.view(torch.int32).item()


def test_counts_treat_any_nonzero_byte_as_routed(mr, orc):
    g = torch.Generator().manual_seed(13)
    T, E = 777, 2304
    vals = torch.tensor([0, 0, 0, 1, 2, 128, 255], dtype=torch.uint8)
    m = vals[torch.randint(0, len(vals), (T, E), generator=g)]
    got = mr.tokens_per_expert(m.cuda())
    torch.cuda.synchronize()
    assert_equal(got, orc.tokens_per_expert(m.numpy()), "tokens_per_expert (0..255 bytes)")


def test_counts_over_long_row_chunks(mr, orc):
    # 2^24 rows of 16 experts: 2048 rows per CTA, 256 per thread, so the
    # byte-wide counters are flushed into the 32-bit ones along the way
    T, E = 1 << 24, 16
    g = torch.Generator().manual_seed(14)
    m = torch.randint(0, 2, (T, E), generator=g, dtype=torch.uint8)
    got = mr.tokens_per_expert(m.cuda())
    torch.cuda.synchronize()
    assert_equal(got, orc.tokens_per_expert(m.numpy()), "tokens_per_expert (long chunks)")
