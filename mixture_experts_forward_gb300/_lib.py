"""ctypes binding of libmoe.so (the C ABI of include/moe.h).

Argument marshalling only: every step runs in the library's CUDA kernels.
There is no fallback — if libmoe.so is missing or cannot be loaded, every
call raises."""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE = 0, 1, 2, 3
MOE_ERR_CUDA, MOE_ERR_TIMEOUT, MOE_ERR_DEVICE_FAULT = 4, 5, 6
DTYPE_FP8, DTYPE_BF16 = 0, 1
EPI_SCATTER, EPI_STORE, EPI_SWIGLU, EPI_STORE_BF16 = 0, 1, 2, 3
SCHED_QUEUE, SCHED_STATIC = 0, 1
CTRL_BYTES = 256

EXPORTS = ["moe_status_string", "moe_num_sms", "moe_route", "moe_layout", "moe_quant_gather",
           "moe_grouped_gemm", "moe_scatter", "moe_workspace_size", "moe_forward",
           "moe_forward_host", "moe_get_error", "moe_debug_set_pipeline_fault", "moe_forward_plan",
           "moe_last_cuda_error", "moe_grouped_gemm_noalloc", "moe_swiglu_quant",
           "moe_forward_workspace_map", "moe_gemm_cta_pairs"]
WS_NONE = (1 << 64) - 1   # MOE_WS_NONE


class MoeError(RuntimeError):
    def __init__(self, code: int, what: str):
        detail = ""
        if code == MOE_ERR_CUDA:
            detail = " — " + lib().moe_last_cuda_error().decode()
        super().__init__(f"{what}: {status_string(code)} ({code}){detail}")
        self.code = code


class GemmArgs(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int), ("epilogue", ctypes.c_int), ("sched", ctypes.c_int),
                ("block_m", ctypes.c_int), ("E", ctypes.c_int), ("N", ctypes.c_int),
                ("K", ctypes.c_int), ("R", ctypes.c_int), ("M", ctypes.c_int),
                ("top_k", ctypes.c_int), ("a", ctypes.c_void_p), ("a_scales", ctypes.c_void_p),
                ("w", ctypes.c_void_p), ("w_scales", ctypes.c_void_p),
                ("offsets", ctypes.c_void_p), ("tile_offsets", ctypes.c_void_p),
                ("sorted_route_ids", ctypes.c_void_p), ("route_weights", ctypes.c_void_p),
                ("out", ctypes.c_void_p), ("k_splits", ctypes.c_int), ("num_ctas", ctypes.c_int),
                ("gather_rows", ctypes.c_int), ("out_scales", ctypes.c_void_p),
                ("cta_pairs", ctypes.c_int)]


class ForwardArgs(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int), ("M", ctypes.c_int), ("K", ctypes.c_int),
                ("N", ctypes.c_int), ("E", ctypes.c_int), ("top_k", ctypes.c_int),
                ("softcap", ctypes.c_float), ("renorm", ctypes.c_int),
                ("logits", ctypes.c_void_p), ("x", ctypes.c_void_p), ("w", ctypes.c_void_p),
                ("w_scales", ctypes.c_void_p), ("w2", ctypes.c_void_p),
                ("block_m", ctypes.c_int), ("sched", ctypes.c_int), ("k_splits", ctypes.c_int),
                ("use_graph", ctypes.c_int), ("gather_rows", ctypes.c_int),
                ("gated", ctypes.c_int), ("w2_scales", ctypes.c_void_p),
                ("cta_pairs", ctypes.c_int)]


class WorkspaceMap(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in
                ("ids", "weights", "counts", "offsets", "tile_offsets", "sorted_route_ids",
                 "route_slot", "a", "a_scales", "h_q", "h_scales")] + \
               [("a_rows", ctypes.c_int), ("block_m", ctypes.c_int)]


_lib = None


def lib():
    """Load libmoe.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m mixture_experts_forward_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        L.moe_status_string.argtypes = [I]
        L.moe_status_string.restype = ctypes.c_char_p
        L.moe_num_sms.restype = I
        L.moe_gemm_cta_pairs.restype = I
        L.moe_last_cuda_error.restype = ctypes.c_char_p
        L.moe_route.argtypes = [P, I, I, I, F, I, P, P, P]
        L.moe_layout.argtypes = [P, I, I, I, I, P, P, P, P, P, P, P]
        L.moe_quant_gather.argtypes = [P, I, I, I, P, P, P, P, I, P]
        L.moe_grouped_gemm.argtypes = [ctypes.POINTER(GemmArgs), P, ctypes.c_size_t, P]
        L.moe_grouped_gemm_noalloc.argtypes = [ctypes.POINTER(GemmArgs), P]
        L.moe_scatter.argtypes = [P, P, P, I, I, I, P, P, P]
        L.moe_swiglu_quant.argtypes = [P, I, I, P, P, P]
        L.moe_workspace_size.argtypes = [ctypes.POINTER(ForwardArgs)]
        L.moe_workspace_size.restype = ctypes.c_size_t
        L.moe_forward.argtypes = [ctypes.POINTER(ForwardArgs), P, P, ctypes.c_size_t, P]
        L.moe_forward_host.argtypes = [ctypes.POINTER(ForwardArgs), P, P, P, P, ctypes.c_size_t, P]
        L.moe_forward_plan.argtypes = [ctypes.POINTER(ForwardArgs), ctypes.POINTER(I),
                                       ctypes.POINTER(I)]
        L.moe_forward_workspace_map.argtypes = [ctypes.POINTER(ForwardArgs),
                                                ctypes.POINTER(WorkspaceMap)]
        L.moe_get_error.argtypes = [P, ctypes.POINTER(ctypes.c_int), P]
        L.moe_debug_set_pipeline_fault.argtypes = [I, ctypes.c_uint64]
        for name in EXPORTS:
            if name not in ("moe_status_string", "moe_num_sms", "moe_workspace_size",
                            "moe_last_cuda_error", "moe_gemm_cta_pairs"):
                getattr(L, name).restype = I
        _lib = L
    return _lib


def status_string(code: int) -> str:
    return lib().moe_status_string(code).decode()


def _check(code: int, what: str):
    if code != MOE_OK:
        raise MoeError(code, what)


def _ptr(t: torch.Tensor | None):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def new_workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """A zeroed device workspace (the control block must start zeroed)."""
    nbytes = max(int(nbytes), CTRL_BYTES)
    return torch.zeros((nbytes + 255) // 256 * 256, dtype=torch.uint8, device=device)


# ------------------------------------------------------------------ steps
def route(logits: torch.Tensor, k: int, softcap: float = 0.0, renorm: int = 1, stream=None):
    M, E = logits.shape
    ids = torch.empty(M, k, dtype=torch.int32, device=logits.device)
    w = torch.empty(M, k, dtype=torch.float32, device=logits.device)
    _check(lib().moe_route(_ptr(logits), M, E, k, float(softcap), int(renorm), _ptr(ids), _ptr(w),
                           _stream(stream)), "moe_route")
    return ids, w


def layout(ids: torch.Tensor, E: int, block_m: int, ws: torch.Tensor, stream=None):
    M, k = ids.shape
    R = M * k
    dev = ids.device
    out = dict(counts=torch.empty(E, dtype=torch.int32, device=dev),
               offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
               sorted_route_ids=torch.empty(R, dtype=torch.int32, device=dev),
               route_slot=torch.empty(R, dtype=torch.int32, device=dev),
               tile_offsets=torch.empty(E + 1, dtype=torch.int32, device=dev))
    _check(lib().moe_layout(_ptr(ids), M, E, k, block_m, _ptr(out["counts"]), _ptr(out["offsets"]),
                            _ptr(out["sorted_route_ids"]), _ptr(out["route_slot"]),
                            _ptr(out["tile_offsets"]), _ptr(ws), _stream(stream)), "moe_layout")
    return out


def quant_gather(x: torch.Tensor, k: int, route_slot: torch.Tensor, zero_acc=None, stream=None):
    M, K = x.shape
    R = M * k
    a_q = torch.empty(R, K, dtype=torch.uint8, device=x.device)
    a_s = torch.empty(K // 128, R, dtype=torch.float32, device=x.device)
    zc = 0 if zero_acc is None else zero_acc.shape[1]
    _check(lib().moe_quant_gather(_ptr(x), M, K, k, _ptr(route_slot), _ptr(a_q), _ptr(a_s),
                                  _ptr(zero_acc), zc, _stream(stream)), "moe_quant_gather")
    return a_q, a_s


def grouped_gemm(*, dtype, epilogue, a, w, offsets, tile_offsets, out, ws, block_m,
                 a_scales=None, w_scales=None, sorted_route_ids=None, route_weights=None,
                 M=0, top_k=0, sched=SCHED_QUEUE, k_splits=0, num_ctas=0, gather_rows=0,
                 out_scales=None, cta_pairs=0, stream=None):
    """moe_grouped_gemm.  gather_rows=1: `a` (and FP8 a_scales) are token-major
    and compact slot s reads row sorted_route_ids[s] // top_k.  FP8 SWIGLU:
    out = u8 [R, N/2] codes of h, out_scales = f32 [N/256, R].  cta_pairs=-1:
    single CTAs only (0: CTA pairs wherever that form exists)."""
    E, N, K = w.shape
    R = sorted_route_ids.numel() if gather_rows else a.shape[0]
    g = GemmArgs(dtype=dtype, epilogue=epilogue, sched=sched, block_m=block_m, E=E, N=N, K=K,
                 R=R, M=M, top_k=top_k, a=a.data_ptr(),
                 a_scales=None if a_scales is None else a_scales.data_ptr(), w=w.data_ptr(),
                 w_scales=None if w_scales is None else w_scales.data_ptr(),
                 offsets=offsets.data_ptr(), tile_offsets=tile_offsets.data_ptr(),
                 sorted_route_ids=None if sorted_route_ids is None else sorted_route_ids.data_ptr(),
                 route_weights=None if route_weights is None else route_weights.data_ptr(),
                 out=out.data_ptr(), k_splits=k_splits, num_ctas=num_ctas,
                 gather_rows=gather_rows,
                 out_scales=None if out_scales is None else out_scales.data_ptr(),
                 cta_pairs=cta_pairs)
    _check(lib().moe_grouped_gemm(ctypes.byref(g), _ptr(ws), ws.numel(), _stream(stream)),
           "moe_grouped_gemm")
    return out


def grouped_gemm_noalloc(*, dtype, epilogue, a, w, offsets, tile_offsets, out, block_m,
                         a_scales=None, w_scales=None, sorted_route_ids=None, route_weights=None,
                         M=0, top_k=0, sched=SCHED_QUEUE, k_splits=0, num_ctas=0,
                         out_scales=None, cta_pairs=0, stream=None):
    """moe_grouped_gemm_noalloc: the same GEMM with the library's own static
    scratch instead of a workspace (for callers that cannot allocate)."""
    E, N, K = w.shape
    g = GemmArgs(dtype=dtype, epilogue=epilogue, sched=sched, block_m=block_m, E=E, N=N, K=K,
                 R=a.shape[0], M=M, top_k=top_k, a=a.data_ptr(),
                 a_scales=None if a_scales is None else a_scales.data_ptr(), w=w.data_ptr(),
                 w_scales=None if w_scales is None else w_scales.data_ptr(),
                 offsets=offsets.data_ptr(), tile_offsets=tile_offsets.data_ptr(),
                 sorted_route_ids=None if sorted_route_ids is None else sorted_route_ids.data_ptr(),
                 route_weights=None if route_weights is None else route_weights.data_ptr(),
                 out=out.data_ptr(), k_splits=k_splits, num_ctas=num_ctas,
                 out_scales=None if out_scales is None else out_scales.data_ptr(),
                 cta_pairs=cta_pairs)
    _check(lib().moe_grouped_gemm_noalloc(ctypes.byref(g), _stream(stream)),
           "moe_grouped_gemm_noalloc")
    return out


def scatter(rows: torch.Tensor, route_slot: torch.Tensor, weights: torch.Tensor,
            ws: torch.Tensor, stream=None):
    """moe_scatter: out bf16 [M, N]; a route with an out-of-range slot records
    MOE_ERR_DEVICE_FAULT in ws's status word (get_error)."""
    M, k = weights.shape
    N = rows.shape[1]
    out = torch.empty(M, N, dtype=torch.bfloat16, device=rows.device)
    _check(lib().moe_scatter(_ptr(rows), _ptr(route_slot), _ptr(weights), M, N, k, _ptr(out),
                             _ptr(ws), _stream(stream)), "moe_scatter")
    return out


def swiglu_quant(gu: torch.Tensor, stream=None):
    """moe_swiglu_quant: gu f32 [R, 2I] (gate columns, then up columns) ->
    (h_q u8 [R, I], h_scales f32 [I/128, R])."""
    R, I2 = gu.shape
    I = I2 // 2
    h_q = torch.empty(R, I, dtype=torch.uint8, device=gu.device)
    h_s = torch.empty(I // 128, R, dtype=torch.float32, device=gu.device)
    _check(lib().moe_swiglu_quant(_ptr(gu), R, I, _ptr(h_q), _ptr(h_s), _stream(stream)),
           "moe_swiglu_quant")
    return h_q, h_s


# ------------------------------------------------------------------ forward
def forward_args(*, dtype, M, K, N, E, top_k, softcap=0.0, renorm=1, logits=None, x=None, w=None,
                 w_scales=None, w2=None, block_m=0, sched=SCHED_QUEUE, k_splits=0,
                 use_graph=1, gather_rows=0, gated=0, w2_scales=None, cta_pairs=0) -> ForwardArgs:
    """Arguments of moe_forward.  gated=1 with dtype FP8: the FP8 gated FFN
    (w = w_up codes [E,2N,K] + w_scales, w2 = w_down codes [E,K,N] + w2_scales).
    cta_pairs=-1: the grouped GEMMs on single CTAs only."""
    return ForwardArgs(dtype=dtype, M=M, K=K, N=N, E=E, top_k=top_k, softcap=float(softcap),
                       renorm=int(renorm), logits=None if logits is None else logits.data_ptr(),
                       x=None if x is None else x.data_ptr(),
                       w=None if w is None else w.data_ptr(),
                       w_scales=None if w_scales is None else w_scales.data_ptr(),
                       w2=None if w2 is None else w2.data_ptr(), block_m=block_m, sched=sched,
                       k_splits=k_splits, use_graph=use_graph, gather_rows=gather_rows,
                       gated=gated,
                       w2_scales=None if w2_scales is None else w2_scales.data_ptr(),
                       cta_pairs=cta_pairs)


def workspace_size(args: ForwardArgs) -> int:
    n = lib().moe_workspace_size(ctypes.byref(args))
    if n == 0:
        raise MoeError(MOE_ERR_INVALID_ARG, "moe_workspace_size")
    return n


def forward_plan(args: ForwardArgs):
    """(block_m, k_splits) that moe_forward uses for these arguments."""
    bm, ks = ctypes.c_int(0), ctypes.c_int(0)
    _check(lib().moe_forward_plan(ctypes.byref(args), ctypes.byref(bm), ctypes.byref(ks)),
           "moe_forward_plan")
    return bm.value, ks.value


def workspace_map(args: ForwardArgs) -> dict:
    """moe_forward_workspace_map: byte offsets of the forward's intermediates
    in its workspace (None for a buffer the forward does not keep), plus
    a_rows and block_m."""
    m = WorkspaceMap()
    _check(lib().moe_forward_workspace_map(ctypes.byref(args), ctypes.byref(m)),
           "moe_forward_workspace_map")
    out = {}
    for name, _ in WorkspaceMap._fields_:
        v = getattr(m, name)
        out[name] = None if (name not in ("a_rows", "block_m") and v == WS_NONE) else v
    return out


def ws_view(ws: torch.Tensor, offset: int, dtype: torch.dtype, shape) -> torch.Tensor:
    """The workspace bytes at ``offset`` viewed as a tensor of dtype/shape
    (no copy)."""
    n = 1
    for s in shape:
        n *= int(s)
    nbytes = n * torch.empty((), dtype=dtype).element_size()
    return ws[offset:offset + nbytes].view(dtype).view(*shape)


def forward(args: ForwardArgs, out: torch.Tensor, ws: torch.Tensor, stream=None):
    _check(lib().moe_forward(ctypes.byref(args), _ptr(out), _ptr(ws), ws.numel(), _stream(stream)),
           "moe_forward")
    return out


def forward_host(args: ForwardArgs, host_logits: torch.Tensor, host_x: torch.Tensor,
                 host_out: torch.Tensor, ws: torch.Tensor, stream=None):
    _check(lib().moe_forward_host(ctypes.byref(args), _ptr(host_logits), _ptr(host_x),
                                  _ptr(host_out), _ptr(ws), ws.numel(), _stream(stream)),
           "moe_forward_host")
    return host_out


def get_error(ws: torch.Tensor, stream=None) -> int:
    st = ctypes.c_int(0)
    _check(lib().moe_get_error(_ptr(ws), ctypes.byref(st), _stream(stream)), "moe_get_error")
    return st.value


def debug_set_pipeline_fault(drop_producer: bool, timeout_ns: int = 0):
    _check(lib().moe_debug_set_pipeline_fault(int(drop_producer), int(timeout_ns)),
           "moe_debug_set_pipeline_fault")


def num_sms() -> int:
    return lib().moe_num_sms()


def gemm_cta_pairs() -> int:
    """CTA pairs resident at once for the FP8 scatter GEMM at block_m 128 (0: not used)."""
    return lib().moe_gemm_cta_pairs()
