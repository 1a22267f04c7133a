"""ctypes binding of libpgg.so: argument marshalling only."""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = None

PAD = 128
FMT_E4M3, FMT_E2M1 = 1, 2
MODE_FWD, MODE_DGRAD, MODE_WGRAD = 0, 1, 2
EPI_NONE, EPI_SWIGLU = 0, 1
_FMT = {"e4m3": FMT_E4M3, "e2m1": FMT_E2M1, FMT_E4M3: FMT_E4M3, FMT_E2M1: FMT_E2M1}

_P, _I64, _I32, _F32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float

# name -> argument types (all return int status)
SIGNATURES = {
    "pgg_version": [],
    "pgg_init": [_I32],
    "pgg_read_error": [_P, _P, _P],
    "pgg_grouped_gemm_fwd": [_P, _P, _P, _P, _I64, _I64, _I64, _I32, _P, _P],
    "pgg_grouped_gemm_dgrad": [_P, _P, _P, _P, _I64, _I64, _I64, _I32, _P, _P],
    "pgg_grouped_gemm_wgrad": [_P, _P, _P, _P, _I64, _I64, _I64, _I32, _P, _P],
    "pgg_grouped_gemm_wgrad_accumulate": [_P, _P, _P, _P, _I64, _I64, _I64, _I32, _P, _P],
    "pgg_grouped_fc1_swiglu": [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I32, _P, _P],
    "pgg_grouped_fc2_dgrad_swiglu_bwd": [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I32, _P, _P],
    "pgg_grouped_fc1_swiglu_clamped": [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I32, _F32, _P, _P],
    "pgg_grouped_fc2_dgrad_swiglu_bwd_clamped": [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I32, _F32, _P, _P],
    "pgg_mx_grouped_gemm_clamped": [_I32, _I32, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I32,
                                    _F32, _P, _P],
    "pgg_mx_quantize_rowwise": [_P, _I64, _I64, _I32, _P, _P, _P],
    "pgg_mx_quantize_rowwise_blocked": [_P, _I64, _I64, _I32, _P, _P, _P],
    "pgg_mx_quantize_colwise": [_P, _I64, _I64, _P, _I32, _I32, _P, _P, _I64, _P, _P],
    "pgg_mx_grouped_gemm": [_I32, _I32, _I32, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64,
                            _I64, _I32, _I64, _P, _P],
    "pgg_moe_permute": [_P, _P, _I64, _I32, _I64, _I32, _P, _P, _P, _P, ctypes.c_size_t, _P, _P],
    "pgg_moe_permute_noalloc": [_P, _P, _I64, _I32, _I64, _I32, _P, _P, _P, _P, _P],
    "pgg_moe_combine": [_P, _P, _P, _P, _I64, _I32, _I64, _P],
    "pgg_fp8_tensor_scale": [_P, _I64, _P, _P],
    "pgg_fp8_quantize_rowwise": [_P, _I64, _I64, _P, _P, _P],
    "pgg_fp8_quantize_colwise": [_P, _I64, _I64, _P, _I32, _P, _P, _I64, _P, _P],
    "pgg_fp8_grouped_gemm": [_I32, _I32, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I32, _I64, _F32, _P,
                             ctypes.c_size_t, _P, _P],
    "pgg_moe_combine_bwd": [_P, _P, _P, _P, _P, _P, _I64, _I32, _I64, _P],
    "pgg_test_stalled_fwd": [_I32, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I32, _I64, ctypes.c_uint64, _P, _P],
}


class PggError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = lib().pgg_status_string(status).decode() if _LIB is not None else str(status)
        super().__init__(f"{where}: pgg status {status} ({msg})")
        self.status = status


def library_path() -> str:
    return os.path.join(_HERE, "libpgg.so")


def lib():
    """Load libpgg.so (raises if it has not been built: there is no fallback)."""
    global _LIB
    if _LIB is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with precision_grouped_gemm_gb300.build.build()")
        L = ctypes.CDLL(path)
        for name, args in SIGNATURES.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = ctypes.c_int
        L.pgg_status_string.argtypes = [ctypes.c_int]
        L.pgg_status_string.restype = ctypes.c_char_p
        L.pgg_moe_permute_workspace_size.argtypes = [_I64, _I32]
        L.pgg_moe_permute_workspace_size.restype = ctypes.c_size_t
        L.pgg_fp8_workspace_size.argtypes = [_I64, _I64, _I32, _I64]
        L.pgg_fp8_workspace_size.restype = ctypes.c_size_t
        _LIB = L
    return _LIB


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(st: int, where: str):
    if st != 0:
        raise PggError(st, where)


def _dev(*ts):
    for t in ts:
        if t is not None:
            if not t.is_cuda:
                raise ValueError("tensors must live on the CUDA device")
            if not t.is_contiguous():
                raise ValueError("tensors must be contiguous")


def _lens(group_lens):
    if group_lens.dtype != torch.int32:
        raise ValueError("group_lens must be int32")
    return group_lens


def version() -> int:
    return lib().pgg_version()


def init(device: int = 0):
    _check(lib().pgg_init(device), "pgg_init")


def read_error(err, stream=None) -> int:
    out = ctypes.c_int32(0)
    _check(lib().pgg_read_error(_ptr(err), ctypes.byref(out), _stream(stream)), "pgg_read_error")
    return out.value


def grouped_gemm_fwd(X, W, group_lens, Y=None, err=None, stream=None):
    """Y_g = X_g . W_g^T; X [M,K] bf16, W [G,N,K] bf16 -> Y [M,N] bf16."""
    M, K = X.shape
    G, N, _ = W.shape
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=X.device)
    _dev(X, W, group_lens, Y, err)
    _check(lib().pgg_grouped_gemm_fwd(_ptr(X), _ptr(W), _ptr(_lens(group_lens)), _ptr(Y), M, N, K, G,
                                      _ptr(err), _stream(stream)), "pgg_grouped_gemm_fwd")
    return Y


def grouped_gemm_dgrad(dY, W, group_lens, dX=None, err=None, stream=None):
    """dX_g = dY_g . W_g; dY [M,N] bf16, W [G,N,K] bf16 -> dX [M,K] bf16."""
    M, N = dY.shape
    G, _, K = W.shape
    if dX is None:
        dX = torch.empty((M, K), dtype=torch.bfloat16, device=dY.device)
    _dev(dY, W, group_lens, dX, err)
    _check(lib().pgg_grouped_gemm_dgrad(_ptr(dY), _ptr(W), _ptr(_lens(group_lens)), _ptr(dX), M, N, K,
                                        G, _ptr(err), _stream(stream)), "pgg_grouped_gemm_dgrad")
    return dX


def grouped_gemm_wgrad(X, dY, group_lens, dW=None, err=None, stream=None):
    """dW_g = dY_g^T . X_g; X [M,K], dY [M,N] bf16 -> dW [G,N,K] bf16 (0 for empty groups)."""
    M, K = X.shape
    N = dY.shape[1]
    G = group_lens.numel()
    if dW is None:
        dW = torch.empty((G, N, K), dtype=torch.bfloat16, device=X.device)
    _dev(X, dY, group_lens, dW, err)
    _check(lib().pgg_grouped_gemm_wgrad(_ptr(X), _ptr(dY), _ptr(_lens(group_lens)), _ptr(dW), M, N, K,
                                        G, _ptr(err), _stream(stream)), "pgg_grouped_gemm_wgrad")
    return dW


def grouped_gemm_wgrad_accumulate(X, dY, group_lens, dW_f32, err=None, stream=None):
    """dW_f32[g] += dY_g^T . X_g in place (fp32 main_grad accumulation); returns dW_f32."""
    M, K = X.shape
    N = dY.shape[1]
    G = group_lens.numel()
    if dW_f32.dtype != torch.float32 or tuple(dW_f32.shape) != (G, N, K):
        raise ValueError("dW_f32 must be float32 [G, N, K]")
    _dev(X, dY, group_lens, dW_f32, err)
    _check(lib().pgg_grouped_gemm_wgrad_accumulate(_ptr(X), _ptr(dY), _ptr(_lens(group_lens)), _ptr(dW_f32), M, N,
                                                   K, G, _ptr(err), _stream(stream)),
           "pgg_grouped_gemm_wgrad_accumulate")
    return dW_f32


def grouped_fc1_swiglu(X, W1, group_lens, A=None, H=None, save_h=True, err=None, stream=None, swiglu_limit=0.0):
    """FC1 + SwiGLU: W1 [G,2I,K] (gate | up) -> A [M,I] and (optionally) H [M,2I];
    swiglu_limit > 0 selects the clamped SwiGLU."""
    M, K = X.shape
    G, I2, _ = W1.shape
    I = I2 // 2
    if A is None:
        A = torch.empty((M, I), dtype=torch.bfloat16, device=X.device)
    if H is None and save_h:
        H = torch.empty((M, 2 * I), dtype=torch.bfloat16, device=X.device)
    _dev(X, W1, group_lens, A, H, err)
    if swiglu_limit:
        _check(lib().pgg_grouped_fc1_swiglu_clamped(_ptr(X), _ptr(W1), _ptr(_lens(group_lens)), _ptr(A), _ptr(H),
                                                    M, I, K, G, swiglu_limit, _ptr(err), _stream(stream)),
               "pgg_grouped_fc1_swiglu_clamped")
    else:
        _check(lib().pgg_grouped_fc1_swiglu(_ptr(X), _ptr(W1), _ptr(_lens(group_lens)), _ptr(A), _ptr(H),
                                            M, I, K, G, _ptr(err), _stream(stream)), "pgg_grouped_fc1_swiglu")
    return A, H


def grouped_fc2_dgrad_swiglu_bwd(dY, W2, H, group_lens, dH=None, err=None, stream=None, swiglu_limit=0.0):
    """dA = dY . W2_g (W2 [G,Hd,I]); dH [M,2I] = SwiGLU backward of dA at the saved H
    (swiglu_limit > 0: of the clamped SwiGLU)."""
    M, Hd = dY.shape
    G, _, I = W2.shape
    if dH is None:
        dH = torch.empty((M, 2 * I), dtype=torch.bfloat16, device=dY.device)
    _dev(dY, W2, H, group_lens, dH, err)
    if swiglu_limit:
        _check(lib().pgg_grouped_fc2_dgrad_swiglu_bwd_clamped(_ptr(dY), _ptr(W2), _ptr(H), _ptr(_lens(group_lens)),
                                                              _ptr(dH), M, Hd, I, G, swiglu_limit, _ptr(err),
                                                              _stream(stream)),
               "pgg_grouped_fc2_dgrad_swiglu_bwd_clamped")
    else:
        _check(lib().pgg_grouped_fc2_dgrad_swiglu_bwd(_ptr(dY), _ptr(W2), _ptr(H), _ptr(_lens(group_lens)),
                                                      _ptr(dH), M, Hd, I, G, _ptr(err), _stream(stream)),
               "pgg_grouped_fc2_dgrad_swiglu_bwd")
    return dH


def mx_quantize_rowwise(x, fmt, codes=None, scales=None, stream=None):
    """bf16 [R,C] -> (codes [R,C] or [R,C/2] u8, scales [R,C/32] u8), blocks along C."""
    R, C = x.shape
    f = _FMT[fmt]
    if codes is None:
        codes = torch.empty((R, C if f == FMT_E4M3 else C // 2), dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty((R, C // 32), dtype=torch.uint8, device=x.device)
    _dev(x, codes, scales)
    _check(lib().pgg_mx_quantize_rowwise(_ptr(x), R, C, f, _ptr(codes), _ptr(scales), _stream(stream)),
           "pgg_mx_quantize_rowwise")
    return codes, scales


def mx_quantize_rowwise_blocked(x, fmt, codes=None, scales=None, stream=None):
    """bf16 [R,C] (C % 128 == 0) -> (codes as mx_quantize_rowwise, scales [round_up(R,128), C/32]
    bytes in the blocked atom layout): the forward GEMM's weight operand."""
    R, C = x.shape
    f = _FMT[fmt]
    if codes is None:
        codes = torch.empty((R, C if f == FMT_E4M3 else C // 2), dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty((-(-R // 128) * 128, C // 32), dtype=torch.uint8, device=x.device)
    _dev(x, codes, scales)
    _check(lib().pgg_mx_quantize_rowwise_blocked(_ptr(x), R, C, f, _ptr(codes), _ptr(scales), _stream(stream)),
           "pgg_mx_quantize_rowwise_blocked")
    return codes, scales


def mx_pad_rows(M: int, G: int) -> int:
    """An M_pad that always holds sum(round_up(len_g, PAD)) for any split of M rows in G groups."""
    return -(-(M + G * (PAD - 1)) // PAD) * PAD


def mx_quantize_colwise(x, group_lens, fmt, M_pad=None, codes_t=None, scales_t=None, err=None,
                        stream=None):
    """bf16 [M,C] + group_lens -> transposed codes_t [C,M_pad] (or [C,M_pad/2]) and scales_t
    [round_up(C,128), M_pad/32] bytes in the blocked atom layout (see pgg.h)."""
    M, C = x.shape
    f = _FMT[fmt]
    G = 1 if group_lens is None else group_lens.numel()
    if M_pad is None:
        M_pad = mx_pad_rows(M, G)
    if codes_t is None:
        codes_t = torch.empty((C, M_pad if f == FMT_E4M3 else M_pad // 2), dtype=torch.uint8, device=x.device)
    if scales_t is None:  # blocked atom layout, rows padded to a multiple of 128
        scales_t = torch.empty((-(-C // 128) * 128, M_pad // 32), dtype=torch.uint8, device=x.device)
    _dev(x, group_lens, codes_t, scales_t, err)
    lens = None if group_lens is None else _lens(group_lens)
    _check(lib().pgg_mx_quantize_colwise(_ptr(x), M, C, _ptr(lens), G, f, _ptr(codes_t), _ptr(scales_t),
                                         M_pad, _ptr(err), _stream(stream)), "pgg_mx_quantize_colwise")
    return codes_t, scales_t


def mx_grouped_gemm(mode, fmt, A, SA, B, SB, group_lens, M, N, K, out=None, out2=None, H=None,
                    epilogue=EPI_NONE, M_pad=0, err=None, stream=None, out_q=None, swiglu_limit=0.0):
    """Block-scaled grouped GEMM on MX operands (see pgg.h for the per-mode layouts).

    out_q: optional (codes, scales) receiving the row-wise MX quantization of `out`
    (SwiGLU epilogues only); swiglu_limit > 0 (SwiGLU epilogues) clamps the SwiGLU."""
    f = _FMT[fmt]
    G = group_lens.numel()
    dev = A.device
    if out is None:
        if mode == MODE_FWD:
            shape = (M, N // 2) if epilogue == EPI_SWIGLU else (M, N)
        elif mode == MODE_DGRAD:
            shape = (M, 2 * K) if epilogue == EPI_SWIGLU else (M, K)
        else:
            shape = (G, N, K)
        out = torch.empty(shape, dtype=torch.bfloat16, device=dev)
    qc, qs = out_q if out_q is not None else (None, None)
    _dev(A, SA, B, SB, group_lens, out, out2, H, err, qc, qs)
    if swiglu_limit:
        if epilogue != EPI_SWIGLU:
            raise ValueError("swiglu_limit needs the SwiGLU epilogue")
        _check(lib().pgg_mx_grouped_gemm_clamped(mode, f, _ptr(A), _ptr(SA), _ptr(B), _ptr(SB), _ptr(H),
                                                 _ptr(_lens(group_lens)), _ptr(out), _ptr(out2), _ptr(qc), _ptr(qs),
                                                 M, N, K, G, swiglu_limit, _ptr(err), _stream(stream)),
               "pgg_mx_grouped_gemm_clamped")
    else:
        _check(lib().pgg_mx_grouped_gemm(mode, f, epilogue, _ptr(A), _ptr(SA), _ptr(B), _ptr(SB), _ptr(H),
                                         _ptr(_lens(group_lens)), _ptr(out), _ptr(out2), _ptr(qc), _ptr(qs), M, N,
                                         K, G, M_pad, _ptr(err), _stream(stream)), "pgg_mx_grouped_gemm")
    return out


def fp8_tensor_scale(x, amax_scale=None, stream=None):
    """bf16 tensor (numel % 8 == 0) -> device float32[2] = (s, amax): amax over the finite
    elements, s = 448 / amax (current scaling, see pgg.h)."""
    if amax_scale is None:
        amax_scale = torch.empty(2, dtype=torch.float32, device=x.device)
    _dev(x, amax_scale)
    _check(lib().pgg_fp8_tensor_scale(_ptr(x), x.numel(), _ptr(amax_scale), _stream(stream)),
           "pgg_fp8_tensor_scale")
    return amax_scale


def fp8_quantize_rowwise(x, amax_scale, codes=None, stream=None):
    """bf16 [R, C] -> e4m3 codes [R, C] (u8) with the tensor scale amax_scale[0]."""
    R, C = x.shape
    if codes is None:
        codes = torch.empty((R, C), dtype=torch.uint8, device=x.device)
    _dev(x, amax_scale, codes)
    _check(lib().pgg_fp8_quantize_rowwise(_ptr(x), R, C, _ptr(amax_scale), _ptr(codes), _stream(stream)),
           "pgg_fp8_quantize_rowwise")
    return codes


def fp8_quantize_colwise(x, group_lens, amax_scale, M_pad=None, codes_t=None, err=None, stream=None):
    """bf16 [M, C] + group_lens -> e4m3 codes_t [C, M_pad] in the group-padded column-wise
    layout (the wgrad operand), with the tensor scale amax_scale[0]."""
    M, C = x.shape
    G = 1 if group_lens is None else group_lens.numel()
    if M_pad is None:
        M_pad = mx_pad_rows(M, G)
    if codes_t is None:
        codes_t = torch.empty((C, M_pad), dtype=torch.uint8, device=x.device)
    _dev(x, group_lens, amax_scale, codes_t, err)
    lens = None if group_lens is None else _lens(group_lens)
    _check(lib().pgg_fp8_quantize_colwise(_ptr(x), M, C, _ptr(lens), G, _ptr(amax_scale), _ptr(codes_t), M_pad,
                                          _ptr(err), _stream(stream)), "pgg_fp8_quantize_colwise")
    return codes_t


def fp8_workspace_size(N: int, K: int, G: int, M_pad: int = 0) -> int:
    return lib().pgg_fp8_workspace_size(N, K, G, M_pad)


def fp8_grouped_gemm(mode, A, scale_a, B, scale_b, group_lens, M, N, K, out=None, out2=None, H=None,
                     epilogue=EPI_NONE, M_pad=0, ws=None, err=None, stream=None, swiglu_limit=0.0):
    """FP8 tensor-wise grouped GEMM: the MX operand layouts and epilogues in e4m3, one scale per
    operand (scale_a / scale_b are the operands' amax_scale tensors; see pgg.h)."""
    G = group_lens.numel()
    dev = A.device
    if out is None:
        if mode == MODE_FWD:
            shape = (M, N // 2) if epilogue == EPI_SWIGLU else (M, N)
        elif mode == MODE_DGRAD:
            shape = (M, 2 * K) if epilogue == EPI_SWIGLU else (M, K)
        else:
            shape = (G, N, K)
        out = torch.empty(shape, dtype=torch.bfloat16, device=dev)
    _dev(A, scale_a, B, scale_b, group_lens, out, out2, H, ws, err)
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(lib().pgg_fp8_grouped_gemm(mode, epilogue, _ptr(A), _ptr(scale_a), _ptr(B), _ptr(scale_b), _ptr(H),
                                      _ptr(_lens(group_lens)), _ptr(out), _ptr(out2), M, N, K, G, M_pad,
                                      swiglu_limit, _ptr(ws), ws_bytes, _ptr(err), _stream(stream)),
           "pgg_fp8_grouped_gemm")
    return out


def moe_permute_workspace_size(T: int, E: int) -> int:
    return int(lib().pgg_moe_permute_workspace_size(T, E))


def moe_permute(topk_ids, X, E, Xs=None, group_lens=None, pos=None, ws=None, err=None, stream=None):
    """topk_ids [T,k] int32 (+ X [T,H] bf16 or None) -> (Xs [T*k,H], group_lens [E], pos [T,k])."""
    T, k = topk_ids.shape
    if topk_ids.dtype != torch.int32:
        raise ValueError("topk_ids must be int32")
    dev = topk_ids.device
    H = 0 if X is None else X.shape[1]
    if X is not None and Xs is None:
        Xs = torch.empty((T * k, H), dtype=torch.bfloat16, device=dev)
    if group_lens is None:
        group_lens = torch.empty(E, dtype=torch.int32, device=dev)
    if pos is None:
        pos = torch.empty((T, k), dtype=torch.int32, device=dev)
    nbytes = moe_permute_workspace_size(T, E)
    if ws is None:
        ws = torch.empty(max(1, nbytes // 4), dtype=torch.int32, device=dev)
    _dev(topk_ids, X, Xs, group_lens, pos, ws, err)
    _check(lib().pgg_moe_permute(_ptr(topk_ids), _ptr(X), T, k, H, E, _ptr(Xs), _ptr(group_lens), _ptr(pos),
                                 _ptr(ws), ws.numel() * ws.element_size(), _ptr(err), _stream(stream)),
           "pgg_moe_permute")
    return Xs, group_lens, pos


def moe_combine(Ys, pos, w=None, out=None, stream=None):
    """out[t] = sum_j w[t,j] * Ys[pos[t,j]] (w None: weight 1, the permute backward)."""
    T, k = pos.shape
    H = Ys.shape[1]
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=Ys.device)
    if w is not None and w.dtype != torch.float32:
        raise ValueError("w must be float32")
    _dev(Ys, pos, w, out)
    _check(lib().pgg_moe_combine(_ptr(Ys), _ptr(pos), _ptr(w), _ptr(out), T, k, H, _stream(stream)),
           "pgg_moe_combine")
    return out


def moe_combine_bwd(dOut, Ys, pos, w, dYs=None, dw=None, stream=None):
    """-> (dYs [R,H] bf16 with dYs[pos[t,j]] = w[t,j] dOut[t], dw [T,k] fp32)."""
    T, k = pos.shape
    H = dOut.shape[1]
    if dYs is None:
        dYs = torch.empty_like(Ys)
    if dw is None:
        dw = torch.empty((T, k), dtype=torch.float32, device=dOut.device)
    if w.dtype != torch.float32:
        raise ValueError("w must be float32")
    _dev(dOut, Ys, pos, w, dYs, dw)
    _check(lib().pgg_moe_combine_bwd(_ptr(dOut), _ptr(Ys), _ptr(pos), _ptr(w), _ptr(dYs), _ptr(dw), T, k, H,
                                     _stream(stream)), "pgg_moe_combine_bwd")
    return dYs, dw
