"""Python binding of libnf4bwd.so: the NF4-dequant-fused backward-A GEMM.

    grad_A[M x K] = grad_out[M x N] @ dequant(B_nf4[K x N])^T

(page "aprender-gpu 0.32.0 -- src/kernels/backward/nf4_tensor_core.rs", struct
doc comment.)  Argument marshalling only: every step runs in the library's CUDA
kernels.  PyTorch provides device memory and the current stream; the functions
enqueue work on ``torch.cuda.current_stream()`` and return without waiting.

There is no fallback: if the compiled library is missing, every call raises.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libnf4bwd.so")

NF4_OK = 0
NF4_ERR_INVALID = 1
NF4_ERR_ALIGN = 2
NF4_ERR_CUDA = 3
NF4_ERR_TIMEOUT = 4
NF4_ERR_WORKSPACE = 5
NF4_F32 = 0
NF4_BF16 = 1
NF4_F16 = 2

# Every function the header declares, with (restype, argtypes).
_vp, _i, _sz = C.c_void_p, C.c_int, C.c_size_t


class Nf4Problem(C.Structure):
    """Mirror of ``nf4_problem``."""
    _fields_ = [("grad_out", _vp), ("go_dtype", _i), ("scales", _vp), ("data", _vp),
                ("grad_A", _vp), ("M", _i), ("N", _i), ("K", _i)]


class Nf4Part(C.Structure):
    """Mirror of ``nf4_part``."""
    _fields_ = [("grad_out", _vp), ("go_dtype", _i), ("N", _i)]


class Nf4FusedProblem(C.Structure):
    """Mirror of ``nf4_fused_problem``."""
    _fields_ = [("parts", C.POINTER(Nf4Part)), ("count", _i), ("scales", _vp), ("data", _vp),
                ("grad_x", _vp), ("M", _i), ("K", _i)]


SIGNATURES = {
    "nf4_abi_version": (_i, []),
    "nf4_status_string": (C.c_char_p, [_i]),
    "nf4_quantize": (_i, [_vp, _i, _i, _vp, _vp, _vp]),
    "nf4_dequantize_f16": (_i, [_vp, _vp, _i, _i, _vp, _vp]),
    "nf4_backward_a": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _vp]),
    "nf4_backward_a_ex": (_i, [_vp, _i, _vp, _vp, _vp, _i, _i, _i, _vp]),
    "nf4_backward_a_ws_bytes": (_sz, [_i, _i]),
    "nf4_backward_a_ws": (_i, [_vp, _i, _vp, _vp, _vp, _i, _i, _i, _vp, _sz, _vp]),
    "nf4_forward_ws_bytes": (_sz, [_i, _i]),
    "rms_norm_backward_ws_bytes": (_sz, [_i, _i]),
    "rms_norm_backward": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _vp, _sz, _vp]),
    "nf4_forward_ws": (_i, [_vp, _i, _vp, _vp, _vp, _i, _i, _i, _vp, _sz, _vp]),
    "nf4_tile_rows": (_i, [_i, _i, _i, _i, _i]),
    "nf4_set_tile_rows": (_i, [_i]),
    "nf4_split_plan": (_i, [_i, _i, _i, C.POINTER(_i), C.POINTER(_i)]),
    "nf4_split_item": (_i, [_i, _i, _i, _i, _i, C.POINTER(_i)]),
    "nf4_backward_a_batched_workspace": (_sz, [_i]),
    "nf4_backward_a_batched_ws_bytes": (_sz, [C.POINTER(Nf4Problem), _i]),
    "nf4_backward_a_batched_ws": (_i, [C.POINTER(Nf4Problem), _i, _vp, _sz, _vp]),
    "nf4_backward_a_batched": (_i, [C.POINTER(Nf4Problem), _i, _vp, _sz, _vp]),
    "nf4_check_error": (_i, [_vp]),
    "nf4_check_error_site": (_i, [_vp, C.POINTER(C.c_uint)]),
    "nf4_backward_a_batched_noalloc": (_i, [C.POINTER(Nf4Problem), _i, _vp]),
    "nf4_set_small_m_max": (_i, [_i]),
    "nf4_small_m_split": (_i, [_i, _i, _i, _i, C.POINTER(_i)]),
    "nf4_watchdog_selftest": (_i, [C.c_longlong, _vp, _vp]),
    "nf4_backward_a_fused": (_i, [C.POINTER(Nf4Part), _i, _vp, _vp, _vp, _i, _i, _vp, _sz, _vp]),
    "nf4_backward_a_fused_batched_ws_bytes": (_sz, [C.POINTER(Nf4FusedProblem), _i]),
    "nf4_backward_a_fused_batched": (_i, [C.POINTER(Nf4FusedProblem), _i, _vp, _sz, _vp]),
    "nf4_gemm_backward_b_splits": (_i, [_i, _i, _i, _i]),
    "nf4_gemm_backward_b_ws_bytes": (_sz, [_i, _i, _i]),
    "nf4_gemm_backward_b": (_i, [_vp, _vp, _i, _vp, _i, _i, _i, _vp, _sz, _vp]),
}

_lib = None


class Nf4Error(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


def lib() -> C.CDLL:
    """The loaded CUDA library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m backward_gemm_gb300.build` (or __graft_entry__.build())")
        L = C.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().nf4_status_string(int(status)).decode()


def _check(rc: int, what: str) -> None:
    if rc != NF4_OK:
        raise Nf4Error(rc, what)


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def _ptr(t: torch.Tensor | None):
    return None if t is None else C.c_void_p(t.data_ptr())


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return NF4_F32
    if t.dtype == torch.bfloat16:
        return NF4_BF16
    if t.dtype == torch.float16:
        return NF4_F16
    raise TypeError(f"grad_out must be float32, bfloat16 or float16, got {t.dtype}")


def _require_cuda_contig(name: str, t: torch.Tensor) -> None:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _check_shapes(go: torch.Tensor, w: "NF4Weight", out: torch.Tensor | None,
                  what: str = "problem") -> tuple[int, int]:
    """Shape and type rules of one backward-A problem: grad_out [M, N] with N =
    the weight's N, the weight's codes [N, K/2] uint8 and scales [N, K/64]
    float32, out (when given) float32 [M, K].  Returns (M, N)."""
    if go.dim() != 2:
        raise ValueError(f"{what}: grad_out must be 2-D [M, N], got shape {tuple(go.shape)}")
    M, N = go.shape
    if N != w.N:
        raise ValueError(f"{what}: grad_out has N={N}, weight has N={w.N}")
    if w.data.dtype != torch.uint8 or w.data.numel() != w.N * (w.K // 2):
        raise ValueError(f"{what}: weight codes must be uint8 [N, K/2] = [{w.N}, {w.K // 2}]")
    if w.scales.dtype != torch.float32 or w.scales.numel() != w.N * (w.K // 64):
        raise ValueError(f"{what}: weight scales must be float32 [N, K/64] = [{w.N}, {w.K // 64}]")
    if out is not None and (out.dtype != torch.float32 or tuple(out.shape) != (M, w.K)):
        raise ValueError(f"{what}: out must be float32 [M, K] = [{M}, {w.K}], got "
                         f"{out.dtype} {tuple(out.shape)}")
    _dtype_code(go)
    return M, N


def _check_devices(go: torch.Tensor, w: "NF4Weight", out: torch.Tensor | None,
                   what: str = "problem") -> None:
    """grad_out, the weight's codes and scales and out (when given): contiguous,
    on one CUDA device."""
    tensors = [("grad_out", go), ("weight codes", w.data), ("weight scales", w.scales)]
    if out is not None:
        tensors.append(("out", out))
    for name, t in tensors:
        _require_cuda_contig(f"{what}: {name}", t)
    if any(t.device != go.device for _, t in tensors):
        raise ValueError(f"{what}: grad_out, the weight and out must be on one device")


def _check_problem(go: torch.Tensor, w: "NF4Weight", out: torch.Tensor | None,
                   what: str = "problem") -> tuple[int, int]:
    """Every rule of one backward-A problem, checked before anything is launched
    (shapes and types first, then devices).  Returns (M, N)."""
    M, N = _check_shapes(go, w, out, what)
    _check_devices(go, w, out, what)
    return M, N


class NF4Weight:
    """A frozen weight B [K x N] in NF4: ``data`` u8 [N, K/2], ``scales`` f32 [N, K/64]."""

    def __init__(self, data: torch.Tensor, scales: torch.Tensor, K: int, N: int):
        self.data, self.scales, self.K, self.N = data, scales, int(K), int(N)

    @property
    def nbytes(self) -> int:
        return self.data.numel() + 4 * self.scales.numel()


def quantize(B: torch.Tensor) -> NF4Weight:
    """Quantise a dense fp32 weight B [K, N] (row-major, on the GPU) to NF4."""
    _require_cuda_contig("B", B)
    if B.dtype != torch.float32 or B.dim() != 2:
        raise ValueError("B must be a 2-D float32 tensor [K, N]")
    K, N = B.shape
    data = torch.empty((N, K // 2), dtype=torch.uint8, device=B.device)
    scales = torch.empty((N, max(K // 64, 1)), dtype=torch.float32, device=B.device)
    _check(lib().nf4_quantize(_ptr(B), K, N, _ptr(data), _ptr(scales), _stream()), "nf4_quantize")
    return NF4Weight(data, scales, K, N)


def dequantize_f16(w: NF4Weight) -> torch.Tensor:
    """deq(B)^T as float16 [N, K] (the GEMM's B^T operand values)."""
    bt = torch.empty((w.N, w.K), dtype=torch.float16, device=w.data.device)
    _check(lib().nf4_dequantize_f16(_ptr(w.scales), _ptr(w.data), w.K, w.N, _ptr(bt), _stream()),
           "nf4_dequantize_f16")
    return bt


def backward_a(grad_out: torch.Tensor, w: NF4Weight, out: torch.Tensor | None = None):
    """grad_A [M, K] fp32 = grad_out [M, N] (fp32 or bf16) @ deq(B)^T."""
    M, N = _check_problem(grad_out, w, out)
    if out is None:
        out = torch.empty((M, w.K), dtype=torch.float32, device=grad_out.device)
    _check(lib().nf4_backward_a_ex(_ptr(grad_out), _dtype_code(grad_out), _ptr(w.scales),
                                   _ptr(w.data), _ptr(out), M, N, w.K, _stream()),
           "nf4_backward_a_ex")
    return out


def ws_workspace(M: int, N: int, device=None, split: bool = True) -> torch.Tensor:
    """Device workspace for :func:`backward_a_ws`: the f16 copy of grad_out and,
    with ``split``, room for splitting a last partial wave of tiles."""
    if split:
        n = int(lib().nf4_backward_a_ws_bytes(M, N))
    else:
        n = 2 * M * ((N + 7) // 8 * 8)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device or "cuda")


def tile_rows(M: int, N: int, K: int, pairs: int, can_split: bool = True) -> int:
    """Tokens per pair tile (256 or 512) the pre-converted path picks (host only)."""
    r = int(lib().nf4_tile_rows(M, N, K, pairs, 1 if can_split else 0))
    if r < 0:
        raise ValueError("invalid tile-rows arguments")
    return r


class tile_rows_forced:
    """Context manager forcing the pre-converted kernel's tile (256 or 512
    tokens; 0 = automatic) within the block."""

    def __init__(self, rows: int):
        self.rows = rows

    def __enter__(self):
        prev = int(lib().nf4_set_tile_rows(int(self.rows)))
        if prev < 0:
            raise ValueError("tile rows must be 0, 256 or 512")
        self.prev = prev
        return self

    def __exit__(self, *exc):
        lib().nf4_set_tile_rows(self.prev)
        return False


def split_plan(tiles: int, stages: int, pairs: int) -> tuple[int, int]:
    """(dp_tiles, sk_tiles) of the ws entry point's split plan (host only)."""
    dp, sk = C.c_int(0), C.c_int(0)
    rc = lib().nf4_split_plan(tiles, stages, pairs, C.byref(dp), C.byref(sk))
    if rc != 0:
        raise ValueError("invalid split-plan arguments")
    return dp.value, sk.value


def split_items(tiles: int, stages: int, pairs: int, pair: int):
    """The items of one pair under the split plan, in run order: tuples
    (tile, s0, s1, first_partner, last_partner)."""
    out = []
    buf = (C.c_int * 5)()
    k = 0
    while True:
        rc = lib().nf4_split_item(tiles, stages, pairs, pair, k, buf)
        if rc < 0:
            raise ValueError("invalid split-item arguments")
        if rc == 0:
            return out
        out.append(tuple(buf))
        k += 1


def backward_a_ws(grad_out: torch.Tensor, w: NF4Weight, workspace: torch.Tensor | None = None,
                  out: torch.Tensor | None = None):
    """As :func:`backward_a`, through ``nf4_backward_a_ws``: grad_out is first
    rounded to f16 into ``workspace`` by its own pass, and the GEMM loads the A
    operand with TMA.  Same result as :func:`backward_a`, bit for bit."""
    M, N = _check_problem(grad_out, w, out)
    if out is None:
        out = torch.empty((M, w.K), dtype=torch.float32, device=grad_out.device)
    if workspace is None:
        workspace = ws_workspace(M, N, grad_out.device)
    _require_cuda_contig("workspace", workspace)
    nbytes = workspace.numel() * workspace.element_size()
    _check(lib().nf4_backward_a_ws(_ptr(grad_out), _dtype_code(grad_out), _ptr(w.scales),
                                   _ptr(w.data), _ptr(out), M, N, w.K, _ptr(workspace), nbytes,
                                   _stream()),
           "nf4_backward_a_ws")
    return out


def forward_ws(A: torch.Tensor, w: NF4Weight, workspace: torch.Tensor | None = None,
               out: torch.Tensor | None = None):
    """C[M, N] = A[M, K] @ dequant(B)[K, N] through ``nf4_forward_ws`` (the
    forward counterpart: contracted over K; A rounded to f16, the same
    dequantised operand values as the backward, f32 accumulation).  A is
    float32, bfloat16 or float16 [M, K]; returns C float32 [M, N]."""
    _require_cuda_contig("A", A)
    M, K = A.shape
    if K != w.K:
        raise ValueError(f"A has K={K}, weight has K={w.K}")
    if out is None:
        out = torch.empty((M, w.N), dtype=torch.float32, device=A.device)
    _require_cuda_contig("out", out)
    if out.dtype != torch.float32 or tuple(out.shape) != (M, w.N):
        raise ValueError("out must be float32 [M, N]")
    if workspace is None:
        n = int(lib().nf4_forward_ws_bytes(M, K))
        workspace = torch.empty(max(n, 256), dtype=torch.uint8, device=A.device)
    _require_cuda_contig("workspace", workspace)
    nbytes = workspace.numel() * workspace.element_size()
    _check(lib().nf4_forward_ws(_ptr(A), _dtype_code(A), _ptr(w.scales), _ptr(w.data), _ptr(out),
                                M, w.N, K, _ptr(workspace), nbytes, _stream()),
           "nf4_forward_ws")
    return out


def rms_norm_backward(x: torch.Tensor, gamma: torch.Tensor, rms: torch.Tensor,
                      grad_y: torch.Tensor, want_gamma: bool = True,
                      workspace: torch.Tensor | None = None, out: torch.Tensor | None = None):
    """Backward of RMS layer normalisation through ``rms_norm_backward``:
    x, grad_y float32 [rows, H], gamma float32 [H], rms float32 [rows] (the
    forward's sqrt(mean(x^2) + eps)).  Returns (grad_x [rows, H], grad_gamma
    [H] or None)."""
    for name, t in (("x", x), ("gamma", gamma), ("rms", rms), ("grad_y", grad_y)):
        _require_cuda_contig(name, t)
        if t.dtype != torch.float32:
            raise TypeError(f"{name} must be float32")
    rows, H = x.shape
    if tuple(grad_y.shape) != (rows, H) or tuple(gamma.shape) != (H,) or tuple(rms.shape) != (rows,):
        raise ValueError("shapes: x, grad_y [rows, H], gamma [H], rms [rows]")
    if out is None:
        out = torch.empty_like(x)
    dgamma = torch.empty(H, dtype=torch.float32, device=x.device) if want_gamma else None
    nbytes = 0
    if want_gamma:
        if workspace is None:
            n = int(lib().rms_norm_backward_ws_bytes(rows, H))
            workspace = torch.empty(max(n, 16), dtype=torch.uint8, device=x.device)
        nbytes = workspace.numel() * workspace.element_size()
    _check(lib().rms_norm_backward(_ptr(x), _ptr(gamma), _ptr(rms), _ptr(grad_y), _ptr(out),
                                   _ptr(dgamma) if want_gamma else None, rows, H,
                                   _ptr(workspace) if want_gamma else None, nbytes, _stream()),
           "rms_norm_backward")
    return out, dgamma


def stack_weights(weights) -> NF4Weight:
    """The NF4 weights of sibling projections (same K) stacked along N, in order:
    their codes and scales concatenated row-wise (the layout
    :func:`backward_a_fused` reads; equal to quantising the concatenated dense
    weights, since every 64-element block lies within one column)."""
    weights = list(weights)
    K = weights[0].K
    if any(w.K != K for w in weights):
        raise ValueError("stacked weights must share K")
    return NF4Weight(torch.cat([w.data for w in weights], 0),
                     torch.cat([w.scales for w in weights], 0), K, sum(w.N for w in weights))


def backward_a_fused(grad_outs, w: NF4Weight, workspace: torch.Tensor | None = None,
                     out: torch.Tensor | None = None):
    """grad_x [M, K] = sum_p grad_outs[p] [M, N_p] @ dequant(B_p)^T in one GEMM
    (``nf4_backward_a_fused``): ``w`` is the projections' weights stacked along
    N (:func:`stack_weights`), ``grad_outs`` their output gradients in the same
    order (float32, bfloat16 or float16; every N_p a multiple of 8)."""
    grad_outs = list(grad_outs)
    if not grad_outs:
        raise ValueError("at least one part")
    M = grad_outs[0].shape[0] if grad_outs[0].dim() == 2 else -1
    for i, g in enumerate(grad_outs):
        if g.dim() != 2 or g.shape[0] != M:
            raise ValueError(f"part {i}: grad_out must be [M, N_p] with M={M}")
        _dtype_code(g)
    if sum(g.shape[1] for g in grad_outs) != w.N:
        raise ValueError(f"the parts' N sum to {sum(g.shape[1] for g in grad_outs)}, "
                         f"the stacked weight has N={w.N}")
    if out is not None and (out.dtype != torch.float32 or tuple(out.shape) != (M, w.K)):
        raise ValueError(f"out must be float32 [M, K] = [{M}, {w.K}]")
    for i, g in enumerate(grad_outs):
        _require_cuda_contig(f"part {i}: grad_out", g)
    for name, t in (("weight codes", w.data), ("weight scales", w.scales)):
        _require_cuda_contig(name, t)
    dev = grad_outs[0].device
    if out is None:
        out = torch.empty((M, w.K), dtype=torch.float32, device=dev)
    _require_cuda_contig("out", out)
    if workspace is None:
        workspace = ws_workspace(M, w.N, dev)
    _require_cuda_contig("workspace", workspace)
    arr = (Nf4Part * len(grad_outs))()
    for i, g in enumerate(grad_outs):
        arr[i] = Nf4Part(g.data_ptr(), _dtype_code(g), g.shape[1])
    nbytes = workspace.numel() * workspace.element_size()
    _check(lib().nf4_backward_a_fused(arr, len(grad_outs), _ptr(w.scales), _ptr(w.data), _ptr(out),
                                      M, w.K, _ptr(workspace), nbytes, _stream()),
           "nf4_backward_a_fused")
    return out


def _fused_array(problems):
    """Host arrays of nf4_fused_problem (and their parts) for (grad_outs, w, out)
    items, every item checked before anything is created."""
    problems = list(problems)
    for i, (gos, w, out) in enumerate(problems):
        gos = list(gos)
        if not gos or len(gos) > 8:
            raise ValueError(f"problem {i}: 1 to 8 parts")
        M = gos[0].shape[0] if gos[0].dim() == 2 else -1
        for j, g in enumerate(gos):
            if g.dim() != 2 or g.shape[0] != M:
                raise ValueError(f"problem {i} part {j}: grad_out must be [M, N_p] with M={M}")
            _dtype_code(g)
            _require_cuda_contig(f"problem {i} part {j}: grad_out", g)
        if sum(g.shape[1] for g in gos) != w.N:
            raise ValueError(f"problem {i}: the parts' N sum to {sum(g.shape[1] for g in gos)}, "
                             f"the stacked weight has N={w.N}")
        if out is not None:
            if out.dtype != torch.float32 or tuple(out.shape) != (M, w.K):
                raise ValueError(f"problem {i}: out must be float32 [M, K] = [{M}, {w.K}]")
            _require_cuda_contig(f"problem {i}: out", out)
        _require_cuda_contig(f"problem {i}: weight codes", w.data)
        _require_cuda_contig(f"problem {i}: weight scales", w.scales)
    arr = (Nf4FusedProblem * max(len(problems), 1))()
    keep, outs = [], []
    for i, (gos, w, out) in enumerate(problems):
        gos = list(gos)
        M = gos[0].shape[0]
        if out is None:
            out = torch.empty((M, w.K), dtype=torch.float32, device=gos[0].device)
        parts = (Nf4Part * len(gos))(*[Nf4Part(g.data_ptr(), _dtype_code(g), g.shape[1])
                                      for g in gos])
        keep.append(parts)
        outs.append(out)
        arr[i] = Nf4FusedProblem(parts, len(gos), w.scales.data_ptr(), w.data.data_ptr(),
                                 out.data_ptr(), M, w.K)
    return arr, keep, outs


def backward_a_fused_batched(problems, workspace: torch.Tensor | None = None):
    """Many fused problems in one grouped launch (``nf4_backward_a_fused_batched``).
    ``problems``: sequence of (grad_outs, stacked NF4Weight, out-or-None); a
    one-part problem is a plain backward-A.  Returns the outputs."""
    problems = list(problems)
    arr, keep, outs = _fused_array(problems)
    if workspace is None:
        n = int(lib().nf4_backward_a_fused_batched_ws_bytes(arr, len(problems)))
        workspace = torch.empty(max(n, 256), dtype=torch.uint8,
                                device=outs[0].device if outs else "cuda")
    _require_cuda_contig("workspace", workspace)
    _check(lib().nf4_backward_a_fused_batched(arr, len(problems), _ptr(workspace),
                                              workspace.numel(), _stream()),
           "nf4_backward_a_fused_batched")
    del keep
    return outs


def gemm_backward_b(A: torch.Tensor, grad_C: torch.Tensor, workspace: torch.Tensor | None = None,
                    out: torch.Tensor | None = None):
    """grad_B [K, N] fp32 = A[M, K]^T @ grad_C[M, N] through ``nf4_gemm_backward_b``
    (the weight gradient of C = A @ B): A and grad_C both bfloat16 or both
    float16, K and N multiples of 8.  A workspace (default: allocated here when
    the call splits the tokens) holds per-split partial sums."""
    if A.dim() != 2 or grad_C.dim() != 2 or A.shape[0] != grad_C.shape[0]:
        raise ValueError("A must be [M, K] and grad_C [M, N] with the same M")
    if A.dtype != grad_C.dtype or A.dtype not in (torch.bfloat16, torch.float16):
        raise TypeError("A and grad_C must both be bfloat16 or both float16")
    M, K = A.shape
    N = grad_C.shape[1]
    if out is not None and (out.dtype != torch.float32 or tuple(out.shape) != (K, N)):
        raise ValueError(f"out must be float32 [K, N] = [{K}, {N}]")
    _require_cuda_contig("A", A)
    _require_cuda_contig("grad_C", grad_C)
    if out is None:
        out = torch.empty((K, N), dtype=torch.float32, device=A.device)
    _require_cuda_contig("out", out)
    if workspace is None:
        n = int(lib().nf4_gemm_backward_b_ws_bytes(M, K, N))
        workspace = torch.empty(max(n, 256), dtype=torch.uint8, device=A.device)
    _require_cuda_contig("workspace", workspace)
    nbytes = workspace.numel() * workspace.element_size()
    _check(lib().nf4_gemm_backward_b(_ptr(A), _ptr(grad_C), _dtype_code(A), _ptr(out), M, K, N,
                                     _ptr(workspace), nbytes, _stream()),
           "nf4_gemm_backward_b")
    return out


def fwd_workspace(M: int, K: int, device=None) -> torch.Tensor:
    """Workspace for :func:`forward_ws` (f16 copy of A plus the split area)."""
    n = int(lib().nf4_forward_ws_bytes(M, K))
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device or "cuda")


def batched_workspace(count: int, device=None) -> torch.Tensor:
    n = int(lib().nf4_backward_a_batched_workspace(count))
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device or "cuda")


def _problem_array(items, make_out: bool):
    """The host array of nf4_problem for a grouped call, every item checked by
    the single-call rules first (nothing is allocated or launched when one
    fails); missing outputs are created when ``make_out``."""
    items = list(items)
    for i, (go, w, out) in enumerate(items):
        _check_shapes(go, w, out, f"item {i}")
        if out is None and not make_out:
            raise ValueError(f"item {i}: every output must be given")
    for i, (go, w, out) in enumerate(items):
        _check_devices(go, w, out, f"item {i}")
    arr = (Nf4Problem * max(len(items), 1))()
    outs = []
    for i, (go, w, out) in enumerate(items):
        M, N = go.shape
        if out is None:
            out = torch.empty((M, w.K), dtype=torch.float32, device=go.device)
        outs.append(out)
        arr[i] = Nf4Problem(go.data_ptr(), _dtype_code(go), w.scales.data_ptr(), w.data.data_ptr(),
                            out.data_ptr(), M, N, w.K)
    return arr, outs


def backward_a_batched(items, workspace: torch.Tensor | None = None):
    """Grouped launch.  ``items``: sequence of (grad_out, NF4Weight, out-or-None).
    Returns the list of outputs."""
    items = list(items)
    arr, outs = _problem_array(items, make_out=True)
    if workspace is None:
        workspace = batched_workspace(len(items), items[0][0].device if items else None)
    _require_cuda_contig("workspace", workspace)
    _check(lib().nf4_backward_a_batched(arr, len(items), _ptr(workspace), workspace.numel(),
                                        _stream()), "nf4_backward_a_batched")
    return outs


def batched_ws_bytes(items) -> int:
    """Bytes of workspace :func:`backward_a_batched_ws` needs for ``items``
    (only the grad_out tensors' shapes and types and the weights' K matter)."""
    items = list(items)
    arr = (Nf4Problem * max(len(items), 1))()
    for i, (go, w, _) in enumerate(items):
        M, N = go.shape
        arr[i] = Nf4Problem(0, _dtype_code(go), 0, 0, 0, M, N, w.K)
    return int(lib().nf4_backward_a_batched_ws_bytes(arr, len(items)))


def batched_ws_workspace(items, device=None) -> torch.Tensor:
    """Workspace for :func:`backward_a_batched_ws` (descriptors and f16 copies)."""
    items = list(items)
    dev = device or (items[0][0].device if items else "cuda")
    return torch.empty(max(batched_ws_bytes(items), 256), dtype=torch.uint8, device=dev)


def backward_a_batched_ws(items, workspace: torch.Tensor | None = None):
    """Grouped launch of the pre-converted path (``nf4_backward_a_batched_ws``):
    f16 copies of every fp32/bf16 grad_out, then one pair-kernel launch over all
    problems.  ``items`` as for :func:`backward_a_batched`; returns the outputs."""
    items = list(items)
    arr, outs = _problem_array(items, make_out=True)
    if workspace is None:
        workspace = batched_ws_workspace(items)
    _require_cuda_contig("workspace", workspace)
    _check(lib().nf4_backward_a_batched_ws(arr, len(items), _ptr(workspace), workspace.numel(),
                                           _stream()), "nf4_backward_a_batched_ws")
    return outs


def backward_a_batched_noalloc(items):
    """Grouped launch that allocates nothing on the device (descriptors kept in a
    fixed array inside the library, at most 256 problems).  ``items`` as for
    backward_a_batched, but every output must be given (no tensor is created)."""
    items = list(items)
    arr, outs = _problem_array(items, make_out=False)
    _check(lib().nf4_backward_a_batched_noalloc(arr, len(items), _stream()),
           "nf4_backward_a_batched_noalloc")
    return outs


def set_small_m_max(m_max: int) -> int:
    """Largest M sent to the few-token kernel (0..64); returns the previous limit."""
    return int(lib().nf4_set_small_m_max(int(m_max)))


class small_m_max:
    """Context manager: ``with small_m_max(0): ...`` runs the block with that limit."""

    def __init__(self, m_max: int):
        self.m_max, self.prev = int(m_max), None

    def __enter__(self):
        self.prev = set_small_m_max(self.m_max)
        return self

    def __exit__(self, *exc):
        set_small_m_max(self.prev)
        return False


def small_m_split(N: int, K: int, sms: int, cta_slots: int) -> tuple[int, int]:
    """(cluster size S, 64-wide N stages per cluster rank) the few-token path picks
    on `sms` SMs that hold `cta_slots` of its CTAs at once."""
    per = C.c_int(0)
    S = lib().nf4_small_m_split(N, K, sms, cta_slots, C.byref(per))
    return int(S), int(per.value)


def watchdog_selftest(limit_cycles: int = 200_000) -> torch.Tensor:
    """Enqueue the bounded-wait self-test (a CTA whose waits give up after
    ``limit_cycles``); returns the 3 device words it writes.  The next
    :func:`check_error` raises for the recorded timeout."""
    where = torch.zeros(3, dtype=torch.int32, device="cuda")
    _check(lib().nf4_watchdog_selftest(int(limit_cycles), _ptr(where), _stream()),
           "nf4_watchdog_selftest")
    return where


def check_error() -> None:
    """Synchronise the current stream and raise if a kernel's bounded wait gave up
    (the message then says which block, thread and barrier)."""
    site = (C.c_uint * 4)()
    rc = lib().nf4_check_error_site(_stream(), site)
    if rc == NF4_ERR_TIMEOUT:
        raise Nf4Error(rc, f"nf4_check_error (first wait that gave up: block {site[0] - 1}, "
                           f"thread {site[1]}, shared address {site[2]:#x}, waiting for {site[3]})")
    _check(rc, "nf4_check_error")
