"""Python binding of the GB300 MoE routing library (libmoe_route.so).

Argument marshalling only: every step of the routing path runs in the library's
CUDA kernels.  Tensors are torch CUDA tensors; the binding passes their data
pointers and the current CUDA stream to the C ABI declared in include/moe_route.h.
There is no CPU fallback: if the shared library is missing or a call fails, an
exception is raised.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe_route.so")

OK = 0
E_INVALID_ARG = -1
E_UNSUPPORTED = -2
E_CUDA = -3
E_WORKSPACE = -4
E_DEVICE_TIMEOUT = -5
E_BAD_ID = -6
F32 = 0
BF16 = 1

_lib = None


class MoeRouteError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {strerror(status)} ({status})")


def load(path: str | None = None):
    """Load libmoe_route.so (built by __graft_entry__.build() or _build.build())."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise ImportError(f"{p} is missing: build it first (python -c 'import __graft_entry__ as g; "
                          f"g.build()')")
    lib = ctypes.CDLL(p)
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.moe_route.argtypes = [P, I, P, I, I, I, I, I, F, I, I, P, P, P, P, P, P]
    lib.moe_route.restype = I
    lib.moe_route_ex.argtypes = [P, I, P, I, I, I, I, I, F, I, I, P, P, P, P, P, P, P]
    lib.moe_route_ex.restype = I
    lib.moe_route_with_layout.argtypes = [P, I, P, I, I, I, I, I, F, I, I, P, P, P, P, P, P, I, P, P, P,
                                          I, P]
    lib.moe_route_with_layout.restype = I
    lib.moe_router_gemm_route.argtypes = [P, P, P, I, I, I, I, I, I, F, I, I, P, P, P, P, P, P, P]
    lib.moe_router_gemm_route.restype = I
    lib.moe_route_quant.argtypes = [P, I, P, I, I, I, I, I, F, I, I, P, I, P, P, P, P, P, P, P, P]
    lib.moe_route_quant.restype = I
    lib.moe_route_host.argtypes = [P, I, P, I, I, I, I, I, F, I, I, P, P, P, P, P, P]
    lib.moe_route_host.restype = I
    lib.moe_route_host_release.argtypes = []
    lib.moe_route_host_release.restype = I
    lib.moe_route_decode_ctas.argtypes = [I]
    lib.moe_route_decode_ctas.restype = I
    lib.moe_route_bins.argtypes = [I, I, I]
    lib.moe_route_bins.restype = I
    lib.moe_route_num_experts.argtypes = [I, I, I, I]
    lib.moe_route_num_experts.restype = I
    lib.moe_route_reserve.argtypes = []
    lib.moe_route_reserve.restype = I
    lib.moe_route_device_status.argtypes = []
    lib.moe_route_device_status.restype = I
    lib.moe_route_sigmoid.argtypes = [P, I, P, I, P]
    lib.moe_route_sigmoid.restype = I
    lib.moe_route_set_path.argtypes = [I]
    lib.moe_route_set_path.restype = I
    lib.moe_route_arm_barrier_timeout.argtypes = [I, I]
    lib.moe_route_arm_barrier_timeout.restype = I
    lib.moe_route_noalloc.argtypes = [P, I, P, I, I, I, I, I, F, I, I, P, P, P, P, P, P, P]
    lib.moe_route_noalloc.restype = I
    lib.moe_route_layout.argtypes = [P, P, P, I, I, I, I, P, P, P, P, I, P]
    lib.moe_route_layout.restype = I
    lib.moe_route_padded_capacity.argtypes = [I, I, I, I]
    lib.moe_route_padded_capacity.restype = I
    lib.moe_route_index.argtypes = [P, I, I, I, P, P, P, P]
    lib.moe_route_index.restype = I
    lib.moe_route_dispatch_counts.argtypes = [P, I, I, P, P, P]
    lib.moe_route_dispatch_counts.restype = I
    lib.moe_route_alltoall_layout.argtypes = [P, I, I, P, P, P, P]
    lib.moe_route_alltoall_layout.restype = I
    lib.moe_route_empty.argtypes = [I, P]
    lib.moe_route_empty.restype = I
    lib.moe_route_strerror.argtypes = [I]
    lib.moe_route_strerror.restype = ctypes.c_char_p
    if path is None:
        _lib = lib
    return lib


def strerror(status: int) -> str:
    try:
        return load().moe_route_strerror(status).decode()
    except ImportError:
        return f"status {status}"


def _check(rc: int, what: str):
    if rc != OK:
        raise MoeRouteError(rc, what)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def decode_ctas(T: int) -> int:
    """CTAs of the routing kernel's launch for T <= 64 rows."""
    n = load().moe_route_decode_ctas(T)
    if n < 0:
        raise MoeRouteError(n, "moe_route_decode_ctas")
    return n


def bins(E: int, k: int, local_count: int) -> int:
    return load().moe_route_bins(E, k, local_count)


def num_experts(E: int, k: int, local_offset: int, local_count: int) -> int:
    return load().moe_route_num_experts(E, k, local_offset, local_count)


def reserve():
    _check(load().moe_route_reserve(), "moe_route_reserve")


def device_status() -> int:
    return load().moe_route_device_status()


def set_path(path: int) -> int:
    rc = load().moe_route_set_path(path)
    if rc < 0:
        raise MoeRouteError(rc, "moe_route_set_path")
    return rc


def alloc_outputs(T: int, E: int, k: int, local_count: int, device, want_ids: bool = False) -> dict:
    NE = bins(E, k, local_count)
    out = dict(packed=torch.empty((T, k), dtype=torch.int32, device=device),
               counts=torch.empty(NE, dtype=torch.int32, device=device),
               offsets=torch.empty(NE + 1, dtype=torch.int32, device=device),
               perm=torch.empty(T * k, dtype=torch.int32, device=device))
    out["ids"] = torch.empty((T, k), dtype=torch.int32, device=device) if want_ids else None
    return out


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return F32
    if t.dtype in (torch.bfloat16, torch.int16, torch.uint16):
        return BF16
    raise TypeError(f"logits must be float32 or bfloat16, got {t.dtype}")


def route(logits: torch.Tensor, bias: torch.Tensor, *, k: int = 16, n_group: int = 8,
          topk_group: int = 4, scale: float = 2.5, local_offset: int = 0, local_count: int = 0,
          out: dict | None = None, want_ids: bool = False, want_inv: bool = False,
          layout_tile: int | None = None, stream=None) -> dict:
    """moe_route on a [T, E] CUDA tensor of router logits (float32 or bfloat16); with
    want_inv (or an "inv_perm" tensor in out) moe_route_ex, which also writes the inverse
    permutation out["inv_perm"]; with layout_tile, moe_route_with_layout, which also writes
    the expert-GEMM layout for that tile: out["padded_offsets"], out["padded_rows"] and
    out["m_indices"] (allocated at the capacity bound when absent)."""
    if not (logits.is_cuda and bias.is_cuda):
        raise ValueError("logits and bias must be CUDA tensors")
    if not logits.is_contiguous() or not bias.is_contiguous() or bias.dtype != torch.float32:
        raise ValueError("logits and bias must be contiguous; bias float32")
    T, E = logits.shape
    if out is None:
        out = alloc_outputs(T, E, k, local_count, logits.device, want_ids)
    if want_inv and out.get("inv_perm") is None:
        out["inv_perm"] = torch.empty(T * k, dtype=torch.int32, device=logits.device)
    if layout_tile is not None:
        NE = out["counts"].numel()
        cap = padded_capacity(T, k, NE, layout_tile)
        for key, n in (("padded_offsets", NE + 1), ("padded_rows", cap), ("m_indices", cap)):
            if out.get(key) is None:
                out[key] = torch.empty(n, dtype=torch.int32, device=logits.device)
        rc = load().moe_route_with_layout(
            _ptr(logits), _dtype_code(logits), _ptr(bias), T, E, k, n_group, topk_group, float(scale),
            local_offset, local_count, _ptr(out["packed"]), _ptr(out["counts"]), _ptr(out["offsets"]),
            _ptr(out["perm"]), _ptr(out.get("ids")), _ptr(out.get("inv_perm")), layout_tile,
            _ptr(out["padded_offsets"]), _ptr(out["padded_rows"]), _ptr(out["m_indices"]),
            out["padded_rows"].numel(), _stream(stream))
        _check(rc, "moe_route_with_layout")
        return out
    if out.get("inv_perm") is not None:
        rc = load().moe_route_ex(_ptr(logits), _dtype_code(logits), _ptr(bias), T, E, k, n_group,
                                 topk_group, float(scale), local_offset, local_count,
                                 _ptr(out["packed"]), _ptr(out["counts"]), _ptr(out["offsets"]),
                                 _ptr(out["perm"]), _ptr(out.get("ids")), _ptr(out["inv_perm"]),
                                 _stream(stream))
        _check(rc, "moe_route_ex")
        return out
    rc = load().moe_route(_ptr(logits), _dtype_code(logits), _ptr(bias), T, E, k, n_group,
                          topk_group, float(scale), local_offset, local_count, _ptr(out["packed"]),
                          _ptr(out["counts"]), _ptr(out["offsets"]), _ptr(out["perm"]),
                          _ptr(out.get("ids")), _stream(stream))
    _check(rc, "moe_route")
    return out


QUANT_MAX_TOKENS = 64


def route_quant(logits: torch.Tensor, bias: torch.Tensor, x: torch.Tensor, *, k: int = 16,
                n_group: int = 8, topk_group: int = 4, scale: float = 2.5, local_offset: int = 0,
                local_count: int = 0, out: dict | None = None, want_ids: bool = False,
                stream=None) -> dict:
    """moe_route_quant: routing of a decode batch (T <= 64) and, in the same launch, the
    MXFP4 codes (out["x_q"], uint8 [T, H / 2]) and E8M0 scales (out["x_scales"], uint8
    [T, H / 32]) of the activations x (bfloat16 [T, H] on the device)."""
    if not (logits.is_cuda and bias.is_cuda and x.is_cuda):
        raise ValueError("logits, bias and x must be CUDA tensors")
    if x.dtype != torch.bfloat16 or not x.is_contiguous() or x.dim() != 2:
        raise ValueError("x must be a contiguous bfloat16 [T, H] tensor")
    T, E = logits.shape
    H = x.shape[1]
    if out is None:
        out = alloc_outputs(T, E, k, local_count, logits.device, want_ids)
    if "x_q" not in out:
        out["x_q"] = torch.empty((T, H // 2), dtype=torch.uint8, device=logits.device)
        out["x_scales"] = torch.empty((T, H // 32), dtype=torch.uint8, device=logits.device)
    rc = load().moe_route_quant(_ptr(logits), _dtype_code(logits), _ptr(bias), T, E, k, n_group,
                                topk_group, float(scale), local_offset, local_count, _ptr(x), H,
                                _ptr(out["x_q"]), _ptr(out["x_scales"]), _ptr(out["packed"]),
                                _ptr(out["counts"]), _ptr(out["offsets"]), _ptr(out["perm"]),
                                _ptr(out.get("ids")), _stream(stream))
    _check(rc, "moe_route_quant")
    return out


def alloc_host_outputs(T: int, E: int, k: int = 16, local_count: int = 0,
                       want_ids: bool = False) -> dict:
    """Page-locked host output buffers for route_host."""
    NE = load().moe_route_bins(E, k, local_count)
    pin = dict(dtype=torch.int32, pin_memory=True)
    out = {"packed": torch.empty((T, k), **pin), "counts": torch.empty(NE, **pin),
           "offsets": torch.empty(NE + 1, **pin), "perm": torch.empty(T * k, **pin)}
    out["ids"] = torch.empty((T, k), **pin) if want_ids else None
    return out


def route_host(logits: torch.Tensor, bias: torch.Tensor, *, k: int = 16, n_group: int = 8,
               topk_group: int = 4, scale: float = 2.5, local_offset: int = 0, local_count: int = 0,
               out: dict | None = None, want_ids: bool = False, stream=None,
               synchronize: bool = True) -> dict:
    """moe_route_host: a [T, E] CPU tensor of router logits (float32 or bfloat16; pinned
    for asynchronous transfer), bias on the device, results in CPU tensors.  With
    synchronize=False the results are valid once the stream has completed the call."""
    if logits.is_cuda or not bias.is_cuda:
        raise ValueError("logits must be a CPU tensor and bias a CUDA tensor")
    if not logits.is_contiguous() or not bias.is_contiguous() or bias.dtype != torch.float32:
        raise ValueError("logits and bias must be contiguous; bias float32")
    T, E = logits.shape
    if out is None:
        out = alloc_host_outputs(T, E, k, local_count, want_ids)
    rc = load().moe_route_host(_ptr(logits), _dtype_code(logits), _ptr(bias), T, E, k, n_group,
                               topk_group, float(scale), local_offset, local_count,
                               _ptr(out["packed"]), _ptr(out["counts"]), _ptr(out["offsets"]),
                               _ptr(out["perm"]), _ptr(out.get("ids")), _stream(stream))
    _check(rc, "moe_route_host")
    if synchronize:
        (stream or torch.cuda.current_stream()).synchronize()
    return out


def route_noalloc(logits: torch.Tensor, bias: torch.Tensor, *, out: dict, status=None,
                  k: int = 16, n_group: int = 8, topk_group: int = 4, scale: float = 2.5,
                  local_offset: int = 0, local_count: int = 0, stream=None) -> dict:
    """moe_route_noalloc: the same routing with scratch in the library's static device
    array, for callers that cannot allocate.  `out` (see alloc_outputs) must be given;
    `status` is an optional one-element int32 CUDA tensor for device-side errors."""
    T, E = logits.shape
    rc = load().moe_route_noalloc(_ptr(logits), _dtype_code(logits), _ptr(bias), T, E, k, n_group,
                                  topk_group, float(scale), local_offset, local_count,
                                  _ptr(out["packed"]), _ptr(out["counts"]), _ptr(out["offsets"]),
                                  _ptr(out["perm"]), _ptr(out.get("ids")), _ptr(status),
                                  _stream(stream))
    _check(rc, "moe_route_noalloc")
    return out


def router_gemm_route(hidden: torch.Tensor, w_router: torch.Tensor, bias: torch.Tensor, *,
                      k: int = 16, n_group: int = 8, topk_group: int = 4, scale: float = 2.5,
                      local_offset: int = 0, local_count: int = 0, want_logits: bool = True,
                      out: dict | None = None, want_ids: bool = False, stream=None) -> dict:
    """moe_router_gemm_route: bf16 hidden [T, H] x router weight [E, H] -> routing."""
    T, H = hidden.shape
    E = w_router.shape[0]
    if out is None:
        out = alloc_outputs(T, E, k, local_count, hidden.device, want_ids)
    if want_logits and out.get("logits") is None:
        out["logits"] = torch.empty((T, E), dtype=torch.float32, device=hidden.device)
    rc = load().moe_router_gemm_route(_ptr(hidden), _ptr(w_router), _ptr(bias), T, H, E, k, n_group,
                                      topk_group, float(scale), local_offset, local_count,
                                      _ptr(out.get("logits")), _ptr(out["packed"]),
                                      _ptr(out["counts"]), _ptr(out["offsets"]), _ptr(out["perm"]),
                                      _ptr(out.get("ids")), _stream(stream))
    _check(rc, "moe_router_gemm_route")
    return out


def padded_capacity(T: int, k: int, NE: int, tile: int) -> int:
    cap = load().moe_route_padded_capacity(T, k, NE, tile)
    if cap < 0:
        raise MoeRouteError(cap, "moe_route_padded_capacity")
    return cap


def route_layout(out: dict, tile: int = 128, *, k: int | None = None, inv: bool = True,
                 padded: bool = True, layout: dict | None = None, stream=None) -> dict:
    """moe_route_layout on the outputs `out` of route() / router_gemm_route(): inverse
    permutation, tile-padded offsets, padded rows and m_indices (device tensors)."""
    T = out["packed"].shape[0]
    k = out["packed"].shape[1] if k is None else k
    NE = out["counts"].numel()
    dev = out["counts"].device
    cap = padded_capacity(T, k, NE, tile)
    if layout is None:
        layout = dict(
            inv_perm=torch.empty(T * k, dtype=torch.int32, device=dev) if inv else None,
            padded_offsets=torch.empty(NE + 1, dtype=torch.int32, device=dev) if padded else None,
            padded_rows=torch.empty(cap, dtype=torch.int32, device=dev) if padded else None,
            m_indices=torch.empty(cap, dtype=torch.int32, device=dev) if padded else None)
    rows = layout.get("padded_rows")
    mind = layout.get("m_indices")
    capacity = (rows.numel() if rows is not None else mind.numel()) if (rows is not None or mind is not None) else 0
    rc = load().moe_route_layout(_ptr(out["counts"]), _ptr(out["offsets"]), _ptr(out["perm"]), T, k,
                                 NE, tile, _ptr(layout.get("inv_perm")),
                                 _ptr(layout.get("padded_offsets")), _ptr(rows), _ptr(mind),
                                 capacity, _stream(stream))
    _check(rc, "moe_route_layout")
    return layout


def route_index(packed: torch.Tensor, NE: int, *, out: dict | None = None, stream=None) -> dict:
    """moe_route_index: counts, offsets and perm of packed values [T, k] (int32, CUDA)."""
    T, k = packed.shape
    if out is None:
        out = dict(counts=torch.empty(NE, dtype=torch.int32, device=packed.device),
                   offsets=torch.empty(NE + 1, dtype=torch.int32, device=packed.device),
                   perm=torch.empty(T * k, dtype=torch.int32, device=packed.device))
    rc = load().moe_route_index(_ptr(packed), T, k, NE, _ptr(out["counts"]), _ptr(out["offsets"]),
                                _ptr(out["perm"]), _stream(stream))
    _check(rc, "moe_route_index")
    return out


def dispatch_counts(offsets: torch.Tensor, num_ranks: int, stream=None) -> dict:
    """moe_route_dispatch_counts on the offsets of a global-id routing."""
    E = offsets.numel() - 1
    dev = offsets.device
    out = dict(send_counts=torch.empty(num_ranks, dtype=torch.int32, device=dev),
               send_offsets=torch.empty(num_ranks + 1, dtype=torch.int32, device=dev))
    rc = load().moe_route_dispatch_counts(_ptr(offsets), E, num_ranks, _ptr(out["send_counts"]),
                                          _ptr(out["send_offsets"]), _stream(stream))
    _check(rc, "moe_route_dispatch_counts")
    return out


def alltoall_layout(matrix: torch.Tensor, rank: int, stream=None) -> dict:
    """moe_route_alltoall_layout: rank's send/receive layout from the counts matrix."""
    R = matrix.shape[0]
    dev = matrix.device
    out = dict(send_displs=torch.empty(R + 1, dtype=torch.int32, device=dev),
               recv_counts=torch.empty(R, dtype=torch.int32, device=dev),
               recv_displs=torch.empty(R + 1, dtype=torch.int32, device=dev))
    rc = load().moe_route_alltoall_layout(_ptr(matrix.contiguous()), R, rank, _ptr(out["send_displs"]),
                                          _ptr(out["recv_counts"]), _ptr(out["recv_displs"]),
                                          _stream(stream))
    _check(rc, "moe_route_alltoall_layout")
    return out


def empty_kernel(ctas: int = 1, stream=None):
    """Launch the empty floor kernel (decode launch shape)."""
    _check(load().moe_route_empty(ctas, _stream(stream)), "moe_route_empty")


def sigmoid(x: torch.Tensor, stream=None) -> torch.Tensor:
    """Step a1 exactly as the routing kernels compute it."""
    s = torch.empty(x.shape, dtype=torch.float32, device=x.device)
    rc = load().moe_route_sigmoid(_ptr(x), _dtype_code(x), _ptr(s), x.numel(), _stream(stream))
    _check(rc, "moe_route_sigmoid")
    return s
