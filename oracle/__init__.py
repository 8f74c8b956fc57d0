"""CPU oracle for the MoE routing path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference legs may import this package. The product path (the CUDA library and
its Python binding) never imports it, and the two share no code.

This module is argument marshalling around ``oracle.c`` (compiled with gcc into
``liboracle.so`` next to it): numpy arrays in, numpy arrays out. All arithmetic
is in the C file.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

SOFTMAX = 0
SIGMOID = 1

_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (no contraction, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
               "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i32, f32 = ctypes.c_int, ctypes.c_float
        lib.orc_expf.argtypes = [f32]
        lib.orc_expf.restype = f32
        lib.orc_sigmoidf.argtypes = [f32]
        lib.orc_sigmoidf.restype = f32
        lib.orc_expf_array.argtypes = [P, P, ctypes.c_size_t]
        lib.orc_sigmoidf_array.argtypes = [P, P, ctypes.c_size_t]
        lib.orc_router_fwd.argtypes = [i32] * 8 + [f32, f32] + [P] * 7
        lib.orc_router_fwd.restype = i32
        lib.orc_aux_scores_fwd.argtypes = [i32] * 4 + [P] * 3
        lib.orc_aux_scores_fwd.restype = i32
        lib.orc_router_bwd.argtypes = [i32] * 4 + [f32] + [P] * 4
        lib.orc_router_bwd.restype = i32
        lib.orc_aux_scores_bwd.argtypes = [i32] * 3 + [P] * 3
        lib.orc_aux_scores_bwd.restype = i32
        lib.orc_sort_capacity.argtypes = [i32] * 4
        lib.orc_sort_capacity.restype = ctypes.c_size_t
        lib.orc_sort.argtypes = [P, P] + [i32] * 4 + [P] * 4
        lib.orc_sort.restype = i32
        i64, f64 = ctypes.c_int64, ctypes.c_double
        lib.orc_tokens_per_expert.argtypes = [i32, i32, P, P]
        lib.orc_tokens_per_expert.restype = i32
        lib.orc_aux_loss_fwd.argtypes = [i32, i32, i32, f64, i64, P, P, P]
        lib.orc_aux_loss_fwd.restype = i32
        lib.orc_aux_loss_bwd.argtypes = [i32, i32, i32, f64, i64, P, f64, P]
        lib.orc_aux_loss_bwd.restype = i32
        lib.orc_near_tie_gaps.argtypes = [i32] * 4 + [P, P, P]
        lib.orc_near_tie_gaps.restype = i32
        _lib = lib
    return _lib


def _p(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=dtype))


class OracleError(RuntimeError):
    pass


def _check(rc: int, what: str) -> int:
    if rc < 0:
        raise OracleError(f"{what}: arguments rejected")
    return rc


def expf(x) -> np.ndarray:
    """The written fp32 exponential, elementwise."""
    lib = _load()
    x = _c(x, np.float32)
    y = np.empty_like(x)
    lib.orc_expf_array(_p(x), _p(y), x.size)
    return y


def sigmoidf(x) -> np.ndarray:
    lib = _load()
    x = _c(x, np.float32)
    y = np.empty_like(x)
    lib.orc_sigmoidf_array(_p(x), _p(y), x.size)
    return y


def router_fwd(logits, topk: int, score_fn: int = SOFTMAX, renorm: int = 0, n_group: int = 0,
               topk_group: int = 0, n_shared: int = 0, scaling: float = 1.0,
               shared_weight: float = 1.0, bias=None) -> dict:
    """Forward over fp32 logits (T x E); returns probs, routing_map, intermediate,
    topk_idx, topk_w (values in float64)."""
    lib = _load()
    x = _c(logits, np.float32)
    T, E = x.shape
    b = None if bias is None else _c(bias, np.float32)
    probs = np.empty((T, E), np.float64)
    rmap = np.empty((T, E), np.uint8)
    inter = np.empty((T, E), np.float64)
    idx = np.empty((T, topk), np.int32)
    w = np.empty((T, topk), np.float64)
    _check(lib.orc_router_fwd(T, E, topk, score_fn, renorm, n_group, topk_group, n_shared,
                              scaling, shared_weight, _p(x), _p(b), _p(probs), _p(rmap),
                              _p(inter), _p(idx), _p(w)), "orc_router_fwd")
    return dict(probs=probs, routing_map=rmap, intermediate=inter, topk_idx=idx, topk_w=w)


def aux_scores_fwd(logits, topk: int, score_fn: int = SOFTMAX) -> dict:
    lib = _load()
    x = _c(logits, np.float32)
    T, E = x.shape
    scores = np.empty((T, E), np.float64)
    rmap = np.empty((T, E), np.uint8)
    _check(lib.orc_aux_scores_fwd(T, E, topk, score_fn, _p(x), _p(scores), _p(rmap)),
           "orc_aux_scores_fwd")
    return dict(scores=scores, routing_map=rmap)


def router_bwd(grad, intermediate, routing_map, score_fn: int = SOFTMAX, renorm: int = 0,
               scaling: float = 1.0) -> np.ndarray:
    lib = _load()
    g = _c(grad, np.float64)
    s = _c(intermediate, np.float64)
    m = _c(routing_map, np.uint8)
    T, E = g.shape
    dx = np.empty((T, E), np.float64)
    _check(lib.orc_router_bwd(T, E, score_fn, renorm, scaling, _p(g), _p(s), _p(m), _p(dx)),
           "orc_router_bwd")
    return dx


def aux_scores_bwd(grad, scores, score_fn: int = SOFTMAX) -> np.ndarray:
    lib = _load()
    g = _c(grad, np.float64)
    s = _c(scores, np.float64)
    T, E = g.shape
    dx = np.empty((T, E), np.float64)
    _check(lib.orc_aux_scores_bwd(T, E, score_fn, _p(g), _p(s), _p(dx)), "orc_aux_scores_bwd")
    return dx


def sort_capacity(T: int, topk: int, E_tot: int, block_m: int) -> int:
    return int(_load().orc_sort_capacity(T, topk, E_tot, block_m))


def sort(topk_idx, topk_w, E_tot: int, block_m: int) -> dict:
    """Returns sorted_token_ids, sorted_weights, expert_ids (each cut to its
    defined length), num_tokens_post_pad and the number of dropped pairs."""
    lib = _load()
    idx = _c(topk_idx, np.int32)
    w = None if topk_w is None else _c(topk_w, np.float32)
    T, k = idx.shape
    cap = sort_capacity(T, k, E_tot, block_m)
    ids = np.full(cap, -1, np.int32)
    sw = np.zeros(cap, np.float32)
    eids = np.full(max(1, -(-cap // block_m)), -1, np.int32)
    npp = np.zeros(1, np.int32)
    dropped = _check(lib.orc_sort(_p(idx), _p(w), T, k, E_tot, block_m, _p(ids), _p(sw), _p(eids),
                                  _p(npp)), "orc_sort")
    n = int(npp[0])
    return dict(sorted_token_ids=ids[:n], sorted_weights=sw[:n], expert_ids=eids[:n // block_m],
                num_tokens_post_pad=n, dropped=dropped)


def tokens_per_expert(routing_map) -> np.ndarray:
    """Per-expert count of routed rows (column counts of a T x E routing map)."""
    lib = _load()
    m = _c(routing_map, np.uint8)
    T, E = m.shape
    out = np.empty(E, np.int32)
    _check(lib.orc_tokens_per_expert(T, E, _p(m), _p(out)), "orc_tokens_per_expert")
    return out


def aux_loss_fwd(probs, tokens_per_expert, topk: int, coeff: float, total_num_tokens: int) -> float:
    """The aux-loss scalar (switch-style load-balancing loss; see oracle.c)."""
    lib = _load()
    p = _c(probs, np.float64)
    T, E = p.shape
    c = _c(tokens_per_expert, np.int32)
    loss = np.empty(1, np.float64)
    _check(lib.orc_aux_loss_fwd(T, E, topk, coeff, total_num_tokens, _p(p), _p(c), _p(loss)), "orc_aux_loss_fwd")
    return float(loss[0])


def aux_loss_bwd(T: int, tokens_per_expert, topk: int, coeff: float, total_num_tokens: int,
                 grad_loss: float) -> np.ndarray:
    """d loss / d probs (T x E)."""
    lib = _load()
    c = _c(tokens_per_expert, np.int32)
    E = c.shape[0]
    g = np.empty((T, E), np.float64)
    _check(lib.orc_aux_loss_bwd(T, E, topk, coeff, total_num_tokens, _p(c), grad_loss, _p(g)),
           "orc_aux_loss_bwd")
    return g


def near_tie_gaps(logits, k_r: int, score_fn: int = SOFTMAX, bias=None) -> np.ndarray:
    """Per token, the gap between the k_r-th and (k_r+1)-th largest selection
    key (computed in double) in fp32 ulps; -1 where k_r >= E. Informational:
    small gaps mark the tokens whose selection another rounding could flip."""
    lib = _load()
    x = _c(logits, np.float32)
    T, E = x.shape
    b = None if bias is None else _c(bias, np.float32)
    gap = np.empty(T, np.float64)
    _check(lib.orc_near_tie_gaps(T, E, k_r, score_fn, _p(x), _p(b), _p(gap)), "orc_near_tie_gaps")
    return gap
