"""Python binding of libmoerouter.so, the GB300 MoE routing library.

Argument marshalling only: every function here passes device pointers, sizes
and the current CUDA stream to the C entry point of the same name (declared in
include/moe_router.h) and turns a non-zero status into an exception. All
arithmetic runs in the library's CUDA kernels; PyTorch supplies device memory
and streams. There is no fallback: without the compiled library, importing
this package raises.

The ``route`` / ``sort`` / ... helpers at the bottom only allocate the output
tensors and call the entry points.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoerouter.so")

MR_OK, MR_EINVAL, MR_EUNSUPPORTED, MR_ECUDA, MR_ERANGE, MR_ETIMEOUT = 0, 1, 2, 3, 4, 5
MR_SOFTMAX, MR_SIGMOID = 0, 1
MR_F32, MR_BF16 = 0, 1
MR_MAX_FUSED_TOKENS = 16
MR_MAX_FUSED_EXPERTS = 1024
MR_MAX_FUSED_TOKENS_SMALL_E = 64
MR_MAX_FUSED_EXPERTS_SMALL = 256



class mr_router_params(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("E", ctypes.c_int32), ("topk", ctypes.c_int32),
                ("score_fn", ctypes.c_int32), ("in_dtype", ctypes.c_int32), ("renorm", ctypes.c_int32),
                ("n_group", ctypes.c_int32), ("topk_group", ctypes.c_int32), ("n_shared", ctypes.c_int32),
                ("scaling", ctypes.c_float), ("shared_weight", ctypes.c_float),
                ("bias", ctypes.c_void_p)]


_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t
_PP = ctypes.POINTER(mr_router_params)
_SIGS = {
    "moe_router_fwd": ([_PP, _P, _P, _P, _P, _P, _P, _P, _P], _I),
    "moe_router_bwd": ([_PP, _P, _P, _P, _P, _P], _I),
    "moe_aux_scores_fwd": ([_I, _I, _I, _I, _I, _P, _P, _P, _P], _I),
    "moe_aux_scores_bwd": ([_I, _I, _I, _P, _P, _P, _P], _I),
    "moe_sort_capacity": ([_I, _I, _I, _I], _SZ),
    "moe_sort_workspace_bytes": ([_I, _I, _I, _I], _SZ),
    "moe_sort": ([_P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _SZ, _P, _P], _I),
    "moe_sort_noalloc": ([_P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P], _I),
    "moe_sort_noalloc_scratch_bytes": ([], _SZ),
    "moe_router_set_wait_test": ([ctypes.c_uint, _I], _I),
    "moe_router_set_launch_overlap": ([_I], _I),
    "moe_router_fused_workspace_bytes": ([_PP, _I], _SZ),
    "moe_router_fused_fwd_sort": ([_PP, _P, _I, _P, _P, _P, _P, _P, _P, _P, _SZ, _P, _P], _I),
    "moe_router_strerror": ([_I], ctypes.c_char_p),
    "moe_router_set_topk_path": ([_I, _I], _I),
    "moe_router_expf": ([_P, _P, _I, _P], _I),
    "moe_router_exp_value": ([_P, _P, _I, _P], _I),
    "moe_router_noop": ([_P], _I),
    "moe_router_device_status": ([_P, _I, _P], _I),
    "moe_router_bwd_dtype": ([_PP, _I, _P, _P, _P, _P, _P], _I),
    "moe_tokens_per_expert": ([_I, _I, _P, _P, _P], _I),
    "moe_aux_loss_workspace_bytes": ([_I, _I], _SZ),
    "moe_aux_loss_fwd": ([_I, _I, _I, ctypes.c_float, ctypes.c_longlong, _P, _P, _P, _P, _SZ, _P], _I),
    "moe_aux_loss_bwd": ([_I, _I, _I, ctypes.c_float, ctypes.c_longlong, _P, _P, _P, _P], _I),
}


class _Lib:
    """The loaded library; loading happens on first use so that the build
    script inside this package can run before the library exists."""

    _cdll = None

    def __getattr__(self, name):
        if _Lib._cdll is None:
            _Lib._cdll = _load()
        return getattr(_Lib._cdll, name)


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with `python -m top_gating_expert_row_gb300.build` "
            "(nvcc, sm_103a). There is no CPU or PyTorch fallback.")
    cdll = ctypes.CDLL(LIB_PATH)
    for name, (args, res) in _SIGS.items():
        f = getattr(cdll, name)
        f.argtypes = args
        f.restype = res
    return cdll


_lib = _Lib()


class MoERouterError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {strerror(code)}")
        self.code = code


def moe_router_strerror(code: int) -> str:
    return _lib.moe_router_strerror(code).decode()


strerror = moe_router_strerror


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to the MoE routing library must be contiguous")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ok(rc: int, where: str) -> int:
    if rc != MR_OK:
        raise MoERouterError(rc, where)
    return rc


@dataclass
class RouterParams:
    T: int
    E: int
    topk: int
    score_fn: int = MR_SOFTMAX
    in_dtype: int = MR_F32
    renorm: int = 0
    n_group: int = 0
    topk_group: int = 0
    n_shared: int = 0
    scaling: float = 1.0
    shared_weight: float = 1.0
    bias: Optional[torch.Tensor] = None

    def c(self) -> mr_router_params:
        return mr_router_params(self.T, self.E, self.topk, self.score_fn, self.in_dtype, self.renorm,
                                self.n_group, self.topk_group, self.n_shared, self.scaling,
                                self.shared_weight, _ptr(self.bias))


def _params(p) -> mr_router_params:
    return p.c() if isinstance(p, RouterParams) else p


# ------------------------------------------------------------------- entry points (same names as the C ABI)


def moe_router_fwd(p, logits, probs=None, routing_map=None, intermediate=None, topk_idx=None,
                   topk_w=None, status=None, stream=None) -> int:
    cp = _params(p)
    return _ok(_lib.moe_router_fwd(ctypes.byref(cp), _ptr(logits), _ptr(probs), _ptr(routing_map),
                                   _ptr(intermediate), _ptr(topk_idx), _ptr(topk_w), _ptr(status),
                                   _stream(stream)),
               "moe_router_fwd")


def moe_router_bwd_dtype(p, grad_dtype, grad_probs, intermediate, routing_map, grad_logits, stream=None) -> int:
    cp = _params(p)
    return _ok(_lib.moe_router_bwd_dtype(ctypes.byref(cp), grad_dtype, _ptr(grad_probs), _ptr(intermediate),
                                         _ptr(routing_map), _ptr(grad_logits), _stream(stream)),
               "moe_router_bwd_dtype")


def moe_router_bwd(p, grad_probs, intermediate, routing_map, grad_logits, stream=None) -> int:
    cp = _params(p)
    return _ok(_lib.moe_router_bwd(ctypes.byref(cp), _ptr(grad_probs), _ptr(intermediate),
                                   _ptr(routing_map), _ptr(grad_logits), _stream(stream)), "moe_router_bwd")


def moe_aux_scores_fwd(T, E, topk, score_fn, in_dtype, logits, scores=None, routing_map=None,
                       stream=None) -> int:
    return _ok(_lib.moe_aux_scores_fwd(T, E, topk, score_fn, in_dtype, _ptr(logits), _ptr(scores),
                                       _ptr(routing_map), _stream(stream)), "moe_aux_scores_fwd")


def moe_aux_scores_bwd(T, E, score_fn, grad_scores, scores, grad_logits, stream=None) -> int:
    return _ok(_lib.moe_aux_scores_bwd(T, E, score_fn, _ptr(grad_scores), _ptr(scores), _ptr(grad_logits),
                                       _stream(stream)), "moe_aux_scores_bwd")


def moe_sort_capacity(T, topk, E_tot, block_m) -> int:
    return int(_lib.moe_sort_capacity(T, topk, E_tot, block_m))


def moe_sort_workspace_bytes(T, topk, E_tot, block_m) -> int:
    return int(_lib.moe_sort_workspace_bytes(T, topk, E_tot, block_m))


def moe_sort(topk_idx, topk_w, T, topk, E_tot, block_m, sorted_token_ids, sorted_weights, expert_ids,
             num_tokens_post_pad, workspace, ws_bytes=None, status=None, stream=None) -> int:
    if ws_bytes is None:
        ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    return _ok(_lib.moe_sort(_ptr(topk_idx), _ptr(topk_w), T, topk, E_tot, block_m, _ptr(sorted_token_ids),
                             _ptr(sorted_weights), _ptr(expert_ids), _ptr(num_tokens_post_pad),
                             _ptr(workspace), ws_bytes, _ptr(status), _stream(stream)), "moe_sort")


def moe_sort_noalloc(topk_idx, topk_w, T, topk, E_tot, block_m, sorted_token_ids, sorted_weights, expert_ids,
                     num_tokens_post_pad, status=None, stream=None) -> int:
    """moe_sort without a workspace: for callers that cannot allocate device
    memory. Its scratch is a fixed device array inside the library (see
    include/moe_router.h); calls that overlap on the GPU race on it."""
    return _ok(_lib.moe_sort_noalloc(_ptr(topk_idx), _ptr(topk_w), T, topk, E_tot, block_m,
                                     _ptr(sorted_token_ids), _ptr(sorted_weights), _ptr(expert_ids),
                                     _ptr(num_tokens_post_pad), _ptr(status), _stream(stream)),
               "moe_sort_noalloc")


def moe_sort_noalloc_scratch_bytes() -> int:
    """Bytes of moe_sort_noalloc's fixed scratch array, as the loaded library has it."""
    return int(_lib.moe_sort_noalloc_scratch_bytes())


def moe_router_fused_workspace_bytes(p, block_m) -> int:
    cp = _params(p)
    return int(_lib.moe_router_fused_workspace_bytes(ctypes.byref(cp), block_m))


def moe_router_fused_fwd_sort(p, logits, block_m, topk_idx, topk_w, sorted_token_ids, sorted_weights,
                              expert_ids, num_tokens_post_pad, workspace=None, ws_bytes=None, status=None,
                              stream=None) -> int:
    cp = _params(p)
    if ws_bytes is None:
        ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    return _ok(_lib.moe_router_fused_fwd_sort(ctypes.byref(cp), _ptr(logits), block_m, _ptr(topk_idx),
                                              _ptr(topk_w), _ptr(sorted_token_ids), _ptr(sorted_weights),
                                              _ptr(expert_ids), _ptr(num_tokens_post_pad), _ptr(workspace),
                                              ws_bytes, _ptr(status), _stream(stream)), "moe_router_fused_fwd_sort")


def moe_router_set_topk_path(select_threshold: int = 8, force_path: int = 0) -> int:
    return _ok(_lib.moe_router_set_topk_path(select_threshold, force_path), "moe_router_set_topk_path")


def moe_router_set_launch_overlap(enable: bool = True) -> int:
    """Programmatic dependent launch of the library's kernels (on by default)."""
    return _ok(_lib.moe_router_set_launch_overlap(1 if enable else 0), "moe_router_set_launch_overlap")


def moe_router_set_wait_test(tries: int = 0, drop_copies: int = 0) -> int:
    """Test hook of the bounded waits (0, 0 restores the defaults)."""
    return _ok(_lib.moe_router_set_wait_test(tries, drop_copies), "moe_router_set_wait_test")


def moe_router_expf(x, y, stream=None) -> int:
    return _ok(_lib.moe_router_expf(_ptr(x), _ptr(y), x.numel(), _stream(stream)), "moe_router_expf")


def moe_router_exp_value(x, y, stream=None) -> int:
    return _ok(_lib.moe_router_exp_value(_ptr(x), _ptr(y), x.numel(), _stream(stream)), "moe_router_exp_value")


def moe_router_noop(stream=None) -> int:
    return _ok(_lib.moe_router_noop(_stream(stream)), "moe_router_noop")


def moe_router_device_status(out, clear: bool = False, stream=None) -> int:
    return _ok(_lib.moe_router_device_status(_ptr(out), 1 if clear else 0, _stream(stream)),
               "moe_router_device_status")


def device_status(clear: bool = False) -> int:
    """The library's device status word on the current device (0 or MR_ETIMEOUT)."""
    out = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe_router_device_status(out, clear)
    return int(out.item())


def moe_tokens_per_expert(T, E, routing_map, tokens_per_expert, stream=None) -> int:
    return _ok(_lib.moe_tokens_per_expert(T, E, _ptr(routing_map), _ptr(tokens_per_expert), _stream(stream)),
               "moe_tokens_per_expert")


def moe_aux_loss_workspace_bytes(T: int, E: int) -> int:
    return int(_lib.moe_aux_loss_workspace_bytes(T, E))


def moe_aux_loss_fwd(T, E, topk, coeff, total_num_tokens, probs, tokens_per_expert, loss, workspace,
                     ws_bytes=None, stream=None) -> int:
    if ws_bytes is None:
        ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    return _ok(_lib.moe_aux_loss_fwd(T, E, topk, coeff, total_num_tokens, _ptr(probs), _ptr(tokens_per_expert),
                                     _ptr(loss), _ptr(workspace), ws_bytes, _stream(stream)), "moe_aux_loss_fwd")


def moe_aux_loss_bwd(T, E, topk, coeff, total_num_tokens, tokens_per_expert, grad_loss, grad_probs,
                     stream=None) -> int:
    return _ok(_lib.moe_aux_loss_bwd(T, E, topk, coeff, total_num_tokens, _ptr(tokens_per_expert),
                                     _ptr(grad_loss), _ptr(grad_probs), _stream(stream)), "moe_aux_loss_bwd")


# ------------------------------------------------------------------- allocating helpers

PATH_AUTO, PATH_ARGMAX, PATH_SELECT = 0, 1, 2


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return MR_F32
    if t.dtype == torch.bfloat16:
        return MR_BF16
    raise TypeError(f"logits must be float32 or bfloat16, got {t.dtype}")


def params_for(logits: torch.Tensor, topk: int, **kw) -> RouterParams:
    T, E = logits.shape
    return RouterParams(T=T, E=E, topk=topk, in_dtype=_dtype_code(logits), **kw)


def route(logits: torch.Tensor, topk: int, dense: bool = True, compact: bool = True, stream=None,
          status: Optional[torch.Tensor] = None, **kw) -> dict:
    """moe_router_fwd with freshly allocated outputs (probs in the logits dtype)."""
    p = params_for(logits, topk, **kw)
    T, E = logits.shape
    dev = logits.device
    out = {}
    if dense:
        out["probs"] = torch.empty(T, E, dtype=logits.dtype, device=dev)
        out["routing_map"] = torch.empty(T, E, dtype=torch.uint8, device=dev)
        out["intermediate"] = torch.empty(T, E, dtype=torch.float32, device=dev)
    if compact:
        out["topk_idx"] = torch.empty(T, topk, dtype=torch.int32, device=dev)
        out["topk_w"] = torch.empty(T, topk, dtype=torch.float32, device=dev)
    moe_router_fwd(p, logits, out.get("probs"), out.get("routing_map"), out.get("intermediate"),
                   out.get("topk_idx"), out.get("topk_w"), status, stream)
    return out


def route_bwd(p: RouterParams, grad_probs, intermediate, routing_map, stream=None) -> torch.Tensor:
    """grad_logits in grad_probs' dtype (fp32, or bf16 for bf16 logits)."""
    if grad_probs.dtype == torch.bfloat16:
        dx = torch.empty(intermediate.shape, dtype=torch.bfloat16, device=intermediate.device)
        moe_router_bwd_dtype(p, MR_BF16, grad_probs, intermediate, routing_map, dx, stream)
        return dx
    dx = torch.empty_like(intermediate)
    moe_router_bwd(p, grad_probs, intermediate, routing_map, dx, stream)
    return dx


def aux_scores(logits: torch.Tensor, topk: int, score_fn: int = MR_SOFTMAX, stream=None) -> dict:
    T, E = logits.shape
    scores = torch.empty(T, E, dtype=torch.float32, device=logits.device)
    rmap = torch.empty(T, E, dtype=torch.uint8, device=logits.device)
    moe_aux_scores_fwd(T, E, topk, score_fn, _dtype_code(logits), logits, scores, rmap, stream)
    return dict(scores=scores, routing_map=rmap)


def aux_scores_bwd(grad, scores, score_fn: int = MR_SOFTMAX, stream=None) -> torch.Tensor:
    T, E = scores.shape
    dx = torch.empty_like(scores)
    moe_aux_scores_bwd(T, E, score_fn, grad, scores, dx, stream)
    return dx


def sort_buffers(T: int, topk: int, E_tot: int, block_m: int, device) -> dict:
    cap = moe_sort_capacity(T, topk, E_tot, block_m)
    return dict(sorted_token_ids=torch.empty(cap, dtype=torch.int32, device=device),
                sorted_weights=torch.empty(cap, dtype=torch.float32, device=device),
                expert_ids=torch.empty(max(1, -(-cap // block_m)), dtype=torch.int32, device=device),
                num_tokens_post_pad=torch.empty(1, dtype=torch.int32, device=device))


def sort(topk_idx: torch.Tensor, topk_w: Optional[torch.Tensor], E_tot: int, block_m: int,
         status: Optional[torch.Tensor] = None, stream=None) -> dict:
    T, k = topk_idx.shape
    out = sort_buffers(T, k, E_tot, block_m, topk_idx.device)
    ws = torch.empty(max(1, moe_sort_workspace_bytes(T, k, E_tot, block_m)), dtype=torch.uint8,
                     device=topk_idx.device)
    moe_sort(topk_idx, topk_w, T, k, E_tot, block_m, out["sorted_token_ids"], out["sorted_weights"],
             out["expert_ids"], out["num_tokens_post_pad"], ws, None, status, stream)
    return out


def fused_route_sort(logits: torch.Tensor, topk: int, block_m: int, compact: bool = True, stream=None,
                     status: Optional[torch.Tensor] = None, **kw) -> dict:
    p = params_for(logits, topk, **kw)
    T, E = logits.shape
    E_tot = E + p.n_shared
    out = sort_buffers(T, topk, E_tot, block_m, logits.device)
    if compact:
        out["topk_idx"] = torch.empty(T, topk, dtype=torch.int32, device=logits.device)
        out["topk_w"] = torch.empty(T, topk, dtype=torch.float32, device=logits.device)
    nb = moe_router_fused_workspace_bytes(p, block_m)
    ws = torch.empty(max(1, nb), dtype=torch.uint8, device=logits.device) if nb else None
    moe_router_fused_fwd_sort(p, logits, block_m, out.get("topk_idx"), out.get("topk_w"),
                              out["sorted_token_ids"], out["sorted_weights"], out["expert_ids"],
                              out["num_tokens_post_pad"], ws, nb, status, stream)
    return out


def header_symbols() -> list[str]:
    """Function names declared in include/moe_router.h."""
    import re

    hdr = os.path.join(os.path.dirname(_HERE), "include", "moe_router.h")
    with open(hdr) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\*?(moe_\w+)\s*\(", text, re.M)))


def tokens_per_expert(routing_map: torch.Tensor, stream=None) -> torch.Tensor:
    """Per-expert count of routed rows of a uint8 [T, E] routing map (int32 [E])."""
    T, E = routing_map.shape
    out = torch.empty(E, dtype=torch.int32, device=routing_map.device)
    moe_tokens_per_expert(T, E, routing_map, out, stream)
    return out


def aux_loss(probs: torch.Tensor, tokens_per_expert: torch.Tensor, topk: int, coeff: float,
             total_num_tokens: int = None, stream=None) -> torch.Tensor:
    """The aux-loss scalar (one fp32 on the device) of fp32 probs [T, E]."""
    T, E = probs.shape
    N = T if total_num_tokens is None else total_num_tokens
    loss = torch.empty(1, dtype=torch.float32, device=probs.device)
    ws = torch.empty(max(1, moe_aux_loss_workspace_bytes(T, E)), dtype=torch.uint8, device=probs.device)
    moe_aux_loss_fwd(T, E, topk, coeff, N, probs, tokens_per_expert, loss, ws, stream=stream)
    return loss


def aux_loss_bwd(grad_loss: torch.Tensor, tokens_per_expert: torch.Tensor, T: int, topk: int, coeff: float,
                 total_num_tokens: int = None, stream=None) -> torch.Tensor:
    """d loss / d probs (fp32 [T, E])."""
    E = tokens_per_expert.numel()
    N = T if total_num_tokens is None else total_num_tokens
    g = torch.empty(T, E, dtype=torch.float32, device=tokens_per_expert.device)
    moe_aux_loss_bwd(T, E, topk, coeff, N, tokens_per_expert, grad_loss, g, stream)
    return g
