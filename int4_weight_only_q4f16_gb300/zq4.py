"""Python binding of the zq4 C ABI (include/zq4.h).

Argument marshalling only: every function checks that the torch tensors it
is given are CUDA, contiguous and large enough, then calls the C entry point
of the same name with their device pointers and the current CUDA stream.
All arithmetic runs in the CUDA library. There is no fallback: if the
library is not built, importing this module raises.

Packed codes may be any 4-byte integer dtype (torch.int32 holding the uint32
bits, or torch.uint32); f16 data is torch.float16; expert ids torch.int32;
router weights torch.float32.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

ZQ4_OK = 0
ZQ4_ERR_NULL = -1
ZQ4_ERR_SHAPE = -2
ZQ4_ERR_ALIGN = -3
ZQ4_ERR_FLAGS = -4
ZQ4_ERR_CUDA = -5
ZQ4_ERR_UNSUPPORTED = -6
ZQ4_ERR_OVERLAP = -7

MOE_GATE_UP_SILU = 1
MOE_DOWN_COMBINE = 2
DEV_BAD_EXPERT_ID = 1
PREP_COPY = 0
PREP_CONCAT_TO_INTERLEAVED = 1
PREP_SEGMENTED = 2

EXPORTS = ("zq4_status_string", "zq4_last_cuda_error", "zq4_version", "zq4_device_errors", "zq4_gemv",
           "zq4_gate_up_silu", "zq4_moe_gemv", "zq4_prepare_weight", "zq4_dequant_f32",
           "zq4_dequant_f16", "zq4_stack_plan_bytes", "zq4_stack_plan_waits", "zq4_stack_plan_init", "zq4_stack_run", "zq4_segmented_bytes", "zq4_stack_plan_init_static", "zq4_stack_plan_set_wait_limit", "zq4_moe_block",
           "zq4_moe_block_work_bytes", "zq4_gemv_seg", "zq4_gate_up_silu_seg",
           "zq4_gemv_argmax", "zq4_gemv_affine", "zq4_gate_up_silu_affine", "zq4_moe_gemv_affine",
           "zq4_add_rmsnorm_work_bytes", "zq4_gemv_add_rmsnorm", "zq4_qkv_rope_append")


class Zq4Error(RuntimeError):
    def __init__(self, fn: str, status: int, lib):
        self.status = status
        msg = lib.zq4_status_string(status).decode()
        if status == ZQ4_ERR_CUDA:
            msg += f" (cudaError {lib.zq4_last_cuda_error()})"
        super().__init__(f"{fn}: {msg}")


def _load():
    path = _build.LIB
    if not os.path.exists(path):
        raise ImportError(
            f"zq4 CUDA library not built ({path} missing): run "
            "`python -m int4_weight_only_q4f16_gb300.build` or __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    P, I = ctypes.c_void_p, ctypes.c_int
    lib.zq4_status_string.argtypes = [I]
    lib.zq4_status_string.restype = ctypes.c_char_p
    lib.zq4_last_cuda_error.restype = I
    lib.zq4_version.restype = I
    lib.zq4_device_errors.argtypes = [P, I]
    lib.zq4_device_errors.restype = I
    sig = {
        "zq4_gemv": [P, P, P, P, I, I, I, P],
        "zq4_gemv_argmax": [P, P, P, P, P, P, P, I, I, I, P],
        "zq4_gate_up_silu": [P, P, P, P, I, I, I, P],
        "zq4_moe_gemv": [P, P, I, P, P, I, I, I, P, P, I, I, P, P],
        "zq4_prepare_weight": [P, P, P, P, I, I, I, P],
        "zq4_dequant_f32": [P, P, P, I, I, P],
        "zq4_dequant_f16": [P, P, P, I, I, P],
        "zq4_stack_plan_bytes": [P, I, I, P],
        "zq4_stack_plan_set_wait_limit": [P, ctypes.c_ulonglong],
        "zq4_moe_block": [P, P, I, P, P, I, I, I, P, P, I, P, ctypes.c_size_t, P, P],
        "zq4_stack_plan_waits": [P, I, I, P, P],
        "zq4_gemv_affine": [P, P, P, P, P, I, I, I, P],
        "zq4_gate_up_silu_affine": [P, P, P, P, P, I, I, I, P],
        "zq4_moe_gemv_affine": [P, P, P, I, P, P, I, I, I, P, P, I, I, P, P],
        "zq4_gemv_add_rmsnorm": [P, P, P, P, P, ctypes.c_float, P, P, P, I, I, I, P],
        "zq4_qkv_rope_append": [P, P, P, I, I, I, I, I, ctypes.c_double, P, P, P, P, P, I, P, P],
        "zq4_stack_plan_init": [P, I, I, P, ctypes.c_size_t, P, P],
        "zq4_stack_run": [P, P],
        "zq4_stack_plan_init_static": [P, I, I, P, P],
        "zq4_gemv_seg": [P, P, P, I, I, I, P],
        "zq4_gate_up_silu_seg": [P, P, P, I, I, I, P],
    }
    lib.zq4_segmented_bytes.argtypes = [I, I]
    lib.zq4_segmented_bytes.restype = ctypes.c_size_t
    lib.zq4_add_rmsnorm_work_bytes.argtypes = [I, I]
    lib.zq4_add_rmsnorm_work_bytes.restype = ctypes.c_size_t
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = I
    return lib


class StackJob(ctypes.Structure):
    """zq4_stack_job."""
    _fields_ = [("wq", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("x", ctypes.c_void_p),
                ("y", ctypes.c_void_p), ("N", ctypes.c_int), ("K", ctypes.c_int), ("gate_up", ctypes.c_int)]


class StackPlanC(ctypes.Structure):
    """zq4_stack_plan."""
    _fields_ = [("dev", ctypes.c_void_p), ("bytes", ctypes.c_size_t), ("n_jobs", ctypes.c_int),
                ("M", ctypes.c_int), ("grid", ctypes.c_int), ("max_k", ctypes.c_int),
                ("max_tiles", ctypes.c_int), ("device", ctypes.c_int), ("engine", ctypes.c_int),
                ("tiles", ctypes.c_int), ("n_pub", ctypes.c_int), ("gen", ctypes.c_int),
                ("min_unit", ctypes.c_int), ("split_tiles", ctypes.c_int), ("part_records", ctypes.c_int),
                ("entries", ctypes.c_int), ("wait_ns", ctypes.c_ulonglong)]


lib = _load()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _ptr(t, name, nbytes, elem=None):
    """Device pointer of t after checking it can hold nbytes."""
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name}: expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: tensor must be contiguous")
    if elem is not None and t.element_size() != elem:
        raise TypeError(f"{name}: expected {elem}-byte elements, got {t.dtype}")
    if t.numel() * t.element_size() < nbytes:
        raise ValueError(f"{name}: holds {t.numel() * t.element_size()} bytes, needs {nbytes}")
    return ctypes.c_void_p(t.data_ptr())


def _check(fn, status):
    if status != ZQ4_OK:
        raise Zq4Error(fn, status, lib)


def _mat(wq, scales, N, K):
    return (_ptr(wq, "wq", N * (K // 8) * 4, 4), _ptr(scales, "scales", N * (K // 32) * 2, 2))


def _mat_affine(wq, scales, biases, N, K):
    gb = N * (K // 64) * 2
    return (_ptr(wq, "wq", N * (K // 8) * 4, 4), _ptr(scales, "scales", gb, 2), _ptr(biases, "biases", gb, 2))


def gemv_affine(wq, scales, biases, x, N, K, y=None, stream=None):
    """y = x @ W^T for W in the MLX affine format (zq4_gemv_affine):
    scales and biases [N, K/64] f16."""
    M = x.numel() // K
    if y is None:
        y = torch.empty((M, N), dtype=torch.float16, device=x.device)
    w, s, b = _mat_affine(wq, scales, biases, N, K)
    _check("zq4_gemv_affine", lib.zq4_gemv_affine(w, s, b, _ptr(x, "x", M * K * 2, 2),
                                                   _ptr(y, "y", M * N * 2, 2), M, N, K, _stream(stream)))
    return y


def gate_up_silu_affine(wq, scales, biases, x, N2, K, h=None, stream=None):
    """h = silu(x Wg^T) * (x Wu^T), interleaved rows, MLX affine format
    (zq4_gate_up_silu_affine)."""
    M = x.numel() // K
    if h is None:
        h = torch.empty((M, N2 // 2), dtype=torch.float16, device=x.device)
    w, s, b = _mat_affine(wq, scales, biases, N2, K)
    _check("zq4_gate_up_silu_affine",
           lib.zq4_gate_up_silu_affine(w, s, b, _ptr(x, "x", M * K * 2, 2), _ptr(h, "h", M * (N2 // 2) * 2, 2),
                                       M, N2, K, _stream(stream)))
    return h


def gemv(wq, scales, x, N, K, y=None, stream=None):
    """y[M, N] = x[M, K] @ dequant(wq, scales)^T (f16 out)."""
    M = x.numel() // K
    if y is None:
        y = torch.empty((M, N), dtype=torch.float16, device=x.device)
    w, s = _mat(wq, scales, N, K)
    _check("zq4_gemv", lib.zq4_gemv(w, s, _ptr(x, "x", M * K * 2, 2), _ptr(y, "y", M * N * 2, 2),
                                    M, N, K, _stream(stream)))
    return y


DEV_BAD_SLOT = 2


def qkv_rope_append(wq, scales, x, K, H, H_kv, D, rope_base, pos, slot, k_cache, v_cache, q_out=None,
                    dev_status=None, stream=None):
    """q_out [M, H*D]: the rotated queries; rotated keys and the values are
    written into k_cache / v_cache [n_slots, H_kv*D] at rows slot[m]
    (zq4_qkv_rope_append). pos, slot: int32 device tensors [M]."""
    M = x.numel() // K
    N = (H + 2 * H_kv) * D
    n_slots = k_cache.numel() // (H_kv * D)
    if q_out is None:
        q_out = torch.empty((M, H * D), dtype=torch.float16, device=x.device)
    w, s = _mat(wq, scales, N, K)
    cb = n_slots * H_kv * D * 2
    _check("zq4_qkv_rope_append", lib.zq4_qkv_rope_append(
        w, s, _ptr(x, "x", M * K * 2, 2), M, K, H, H_kv, D, float(rope_base), _ptr(pos, "pos", M * 4, 4),
        _ptr(slot, "slot", M * 4, 4), _ptr(q_out, "q_out", M * H * D * 2, 2), _ptr(k_cache, "k_cache", cb, 2),
        _ptr(v_cache, "v_cache", cb, 2), n_slots, _ptr(dev_status, "dev_status", 4, 4), _stream(stream)))
    return q_out


def add_rmsnorm_work_bytes(M, N):
    return int(lib.zq4_add_rmsnorm_work_bytes(M, N))


def gemv_add_rmsnorm(wq, scales, x, resid, gamma, eps, N, K, res_out=None, out=None, work=None, stream=None):
    """(res_out, out): res_out = f16(resid + x W^T), out = f16(RMSNorm(that) *
    gamma) (zq4_gemv_add_rmsnorm). ``work``: a zeroed uint8 device tensor of
    add_rmsnorm_work_bytes(M, N) bytes, reusable across calls (made here if
    not given)."""
    M = x.numel() // K
    if res_out is None:
        res_out = torch.empty((M, N), dtype=torch.float16, device=x.device)
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=x.device)
    wb = add_rmsnorm_work_bytes(M, N)
    if work is None:
        work = torch.zeros(wb, dtype=torch.uint8, device=x.device)
    w, s = _mat(wq, scales, N, K)
    _check("zq4_gemv_add_rmsnorm", lib.zq4_gemv_add_rmsnorm(
        w, s, _ptr(x, "x", M * K * 2, 2), _ptr(resid, "resid", M * N * 2, 2), _ptr(gamma, "gamma", N * 2, 2),
        float(eps), _ptr(res_out, "res_out", M * N * 2, 2), _ptr(out, "out", M * N * 2, 2),
        _ptr(work, "work", wb), M, N, K, _stream(stream)))
    return res_out, out


def gemv_argmax(wq, scales, x, N, K, y32=None, logits=True, maxval=None, idx=None, work=None, stream=None):
    """LM-head step: fp32 logits y32[M, N] (unless logits=False) and, per
    token, the index of the largest logit (lowest index on ties) and that
    logit. Returns (idx int32 [M], maxval float32 [M], y32 or None). A given
    `work` (int64 [M + 8]) must be all zero before its first call; every
    call leaves it zero."""
    M = x.numel() // K
    dev = x.device
    if logits and y32 is None:
        y32 = torch.empty((M, N), dtype=torch.float32, device=dev)
    if idx is None:
        idx = torch.empty((M,), dtype=torch.int32, device=dev)
    if maxval is None:
        maxval = torch.empty((M,), dtype=torch.float32, device=dev)
    if work is None:
        work = torch.zeros((M + 8,), dtype=torch.int64, device=dev)   # zero before the first call
    w, s = _mat(wq, scales, N, K)
    _check("zq4_gemv_argmax",
           lib.zq4_gemv_argmax(w, s, _ptr(x, "x", M * K * 2, 2), _ptr(y32, "y32", M * N * 4, 4) if logits else None,
                               _ptr(idx, "idx", M * 4, 4), _ptr(maxval, "maxval", M * 4, 4),
                               _ptr(work, "work", (M + 8) * 8, 8), M, N, K, _stream(stream)))
    return idx, maxval, (y32 if logits else None)


def gate_up_silu(wq, scales, x, N2, K, h=None, stream=None):
    """h[M, N2/2] = silu(g) * u over interleaved gate/up rows."""
    M = x.numel() // K
    if h is None:
        h = torch.empty((M, N2 // 2), dtype=torch.float16, device=x.device)
    w, s = _mat(wq, scales, N2, K)
    _check("zq4_gate_up_silu",
           lib.zq4_gate_up_silu(w, s, _ptr(x, "x", M * K * 2, 2),
                                _ptr(h, "h", M * (N2 // 2) * 2, 2), M, N2, K, _stream(stream)))
    return h


def moe_gemv(wq_bank, scales_bank, num_experts, x, N, K, expert_ids, mode, route_w=None,
             y=None, dev_status=None, stream=None):
    """Expert-gather GEMV; see zq4_moe_gemv in include/zq4.h for the modes."""
    T, top_k = expert_ids.shape
    if mode == MOE_GATE_UP_SILU:
        xrows, yshape = T, (T, top_k, N // 2)
    else:
        xrows, yshape = T * top_k, (T, N)
    if y is None:
        y = torch.empty(yshape, dtype=torch.float16, device=x.device)
    ybytes = 2
    for d in yshape:
        ybytes *= d
    w = _ptr(wq_bank, "wq_bank", num_experts * N * (K // 8) * 4, 4)
    s = _ptr(scales_bank, "scales_bank", num_experts * N * (K // 32) * 2, 2)
    _check("zq4_moe_gemv", lib.zq4_moe_gemv(
        w, s, num_experts, _ptr(x, "x", xrows * K * 2, 2), _ptr(y, "y", ybytes, 2), T, N, K,
        _ptr(expert_ids, "expert_ids", T * top_k * 4, 4),
        _ptr(route_w, "route_w", T * top_k * 4, 4), top_k, mode,
        _ptr(dev_status, "dev_status", 4, 4), _stream(stream)))
    return y


def moe_block_work_bytes(T, top_k, D, I):
    lib.zq4_moe_block_work_bytes.restype = ctypes.c_size_t
    lib.zq4_moe_block_work_bytes.argtypes = [ctypes.c_int] * 4
    return int(lib.zq4_moe_block_work_bytes(T, top_k, D, I))


def moe_block(gu_seg, dn_seg, num_experts, x, D, I, expert_ids, route_w, y=None, work=None, dev_status=None,
              stream=None):
    """The MoE block in one call (zq4_moe_block): gate_up + SiLU*mul and
    down + weighted combine, each touched expert read once per stage. The
    banks in the segmented layout (prepare_weight(..., PREP_SEGMENTED) over
    all of a bank's rows). Returns (y [T, D] f16, work); see include/zq4.h
    for work's layout (the grouping, then h and z)."""
    T, top_k = expert_ids.shape
    E = num_experts
    wb = moe_block_work_bytes(T, top_k, D, I)
    if y is None:
        y = torch.empty((T, D), dtype=torch.float16, device=x.device)
    if work is None:
        work = torch.zeros(wb, dtype=torch.uint8, device=x.device)
    _check("zq4_moe_block", lib.zq4_moe_block(
        _ptr(gu_seg, "gu_seg", E * segmented_bytes(2 * I, D)), _ptr(dn_seg, "dn_seg", E * segmented_bytes(D, I)),
        E, _ptr(x, "x", T * D * 2, 2), _ptr(y, "y", T * D * 2, 2), T, D, I,
        _ptr(expert_ids, "expert_ids", T * top_k * 4, 4), _ptr(route_w, "route_w", T * top_k * 4, 4), top_k,
        _ptr(work, "work", wb), wb, _ptr(dev_status, "dev_status", 4, 4), _stream(stream)))
    return y, work


def moe_block_views(work, T, top_k, D, I):
    """(grouping ints, h [T, top_k, I] f16, z [T, top_k, D] fp32) inside a
    moe_block work buffer."""
    P = T * top_k
    g_ints = 3 * P + 3
    h_off = (g_ints * 4 + 255) // 256 * 256
    z_off = h_off + (P * I * 2 + 255) // 256 * 256
    group = work[:g_ints * 4].view(torch.int32)
    h = work[h_off:h_off + P * I * 2].view(torch.float16).view(T, top_k, I)
    z = work[z_off:z_off + P * D * 4].view(torch.float32).view(T, top_k, D)
    return group, h, z


def moe_gemv_affine(wq_bank, scales_bank, biases_bank, num_experts, x, N, K, expert_ids, mode, route_w=None,
                    y=None, dev_status=None, stream=None):
    """moe_gemv on affine expert banks (zq4_moe_gemv_affine): scales and
    biases [num_experts * N, K/64] f16."""
    T, top_k = expert_ids.shape
    if mode == MOE_GATE_UP_SILU:
        xrows, yshape = T, (T, top_k, N // 2)
    else:
        xrows, yshape = T * top_k, (T, N)
    if y is None:
        y = torch.empty(yshape, dtype=torch.float16, device=x.device)
    ybytes = 2
    for d in yshape:
        ybytes *= d
    gb = num_experts * N * (K // 64) * 2
    _check("zq4_moe_gemv_affine", lib.zq4_moe_gemv_affine(
        _ptr(wq_bank, "wq_bank", num_experts * N * (K // 8) * 4, 4), _ptr(scales_bank, "scales_bank", gb, 2),
        _ptr(biases_bank, "biases_bank", gb, 2), num_experts, _ptr(x, "x", xrows * K * 2, 2),
        _ptr(y, "y", ybytes, 2), T, N, K, _ptr(expert_ids, "expert_ids", T * top_k * 4, 4),
        _ptr(route_w, "route_w", T * top_k * 4, 4), top_k, mode,
        _ptr(dev_status, "dev_status", 4, 4), _stream(stream)))
    return y


def gemv_seg(wseg, x, N, K, y=None, stream=None):
    """gemv on a segmented-layout matrix (prepare_weight with PREP_SEGMENTED)."""
    M = x.numel() // K
    if y is None:
        y = torch.empty((M, N), dtype=torch.float16, device=x.device)
    _check("zq4_gemv_seg", lib.zq4_gemv_seg(_ptr(wseg, "wseg", segmented_bytes(N, K)), _ptr(x, "x", M * K * 2, 2),
                                            _ptr(y, "y", M * N * 2, 2), M, N, K, _stream(stream)))
    return y


def gate_up_silu_seg(wseg, x, N2, K, h=None, stream=None):
    """gate_up_silu on a segmented-layout matrix."""
    M = x.numel() // K
    if h is None:
        h = torch.empty((M, N2 // 2), dtype=torch.float16, device=x.device)
    _check("zq4_gate_up_silu_seg",
           lib.zq4_gate_up_silu_seg(_ptr(wseg, "wseg", segmented_bytes(N2, K)), _ptr(x, "x", M * K * 2, 2),
                                    _ptr(h, "h", M * (N2 // 2) * 2, 2), M, N2, K, _stream(stream)))
    return h


def segmented_bytes(N, K):
    return int(lib.zq4_segmented_bytes(N, K))


def prepare_weight(wq_src, scales_src, N, K, flags=PREP_CONCAT_TO_INTERLEAVED, wq_dst=None,
                   scales_dst=None, stream=None):
    """Rewrite a matrix into a kernel layout. With PREP_SEGMENTED the result
    is one uint8 tensor of segmented_bytes(N, K) (scales inside) and None."""
    if flags & PREP_SEGMENTED:
        nb = segmented_bytes(N, K)
        if nb == 0:
            raise ValueError("segmented layout needs N > 0 and K % 256 == 0")
        if wq_dst is None:
            wq_dst = torch.empty(nb, dtype=torch.uint8, device=wq_src.device)
        w, s = _mat(wq_src, scales_src, N, K)
        _check("zq4_prepare_weight", lib.zq4_prepare_weight(w, s, _ptr(wq_dst, "wq_dst", nb), None, N, K, flags,
                                                            _stream(stream)))
        return wq_dst, None
    if wq_dst is None:
        wq_dst = torch.empty_like(wq_src)
    if scales_dst is None:
        scales_dst = torch.empty_like(scales_src)
    w, s = _mat(wq_src, scales_src, N, K)
    wd, sd = _mat(wq_dst, scales_dst, N, K)
    _check("zq4_prepare_weight", lib.zq4_prepare_weight(w, s, wd, sd, N, K, flags, _stream(stream)))
    return wq_dst, scales_dst


def dequant_f32(wq, scales, N, K, out=None, stream=None):
    if out is None:
        out = torch.empty((N, K), dtype=torch.float32, device=wq.device)
    w, s = _mat(wq, scales, N, K)
    _check("zq4_dequant_f32", lib.zq4_dequant_f32(w, s, _ptr(out, "w", N * K * 4, 4), N, K,
                                                  _stream(stream)))
    return out


def dequant_f16(wq, scales, N, K, out=None, stream=None):
    if out is None:
        out = torch.empty((N, K), dtype=torch.float16, device=wq.device)
    w, s = _mat(wq, scales, N, K)
    _check("zq4_dequant_f16", lib.zq4_dequant_f16(w, s, _ptr(out, "w", N * K * 2, 2), N, K,
                                                  _stream(stream)))
    return out


DEVERR_WAIT_TIMEOUT = 1          # ZQ4_DEVERR_WAIT_TIMEOUT


def device_errors(clear: bool = True) -> int:
    """Device error word (ZQ4_DEVERR_* bits); synchronises the device."""
    v = ctypes.c_uint32(0)
    _check("zq4_device_errors", lib.zq4_device_errors(ctypes.byref(v), int(clear)))
    return int(v.value)


def status_string(status: int) -> str:
    return lib.zq4_status_string(status).decode()


def stack_plan_waits(jobs, M):
    """zq4_stack_plan_waits on addresses: ``jobs`` is a list of (wq, x, y, N,
    K, gate_up) with plain integer addresses (nothing is read at them).
    Returns (order, dep): the run order as indices of ``jobs``, and per job
    the job it waits for (-1: none)."""
    n = len(jobs)
    arr = (StackJob * n)()
    for i, (wq, x, y, N, K, gate_up) in enumerate(jobs):
        arr[i] = StackJob(wq, None, x, y, N, K, 1 if gate_up else 0)
    order, dep = (ctypes.c_int * n)(), (ctypes.c_int * n)()
    _check("zq4_stack_plan_waits", lib.zq4_stack_plan_waits(ctypes.cast(arr, ctypes.c_void_p), n, M, order, dep))
    return list(order), list(dep)


class StackPlan:
    """A decode step as one launch (zq4_stack_plan_init / zq4_stack_run).

    ``jobs`` is a list of (seg, x, y, N, K, gate_up) with torch CUDA tensors,
    seg the matrix in the segmented layout (prepare_weight with
    PREP_SEGMENTED); a job may take an earlier job's y as its x. The plan keeps
    references to every tensor (they must stay allocated) and owns its
    device buffer."""

    def __init__(self, jobs, M, stream=None):
        arr = (StackJob * len(jobs))()
        self._keep = []
        for i, (seg, x, y, N, K, gate_up) in enumerate(jobs):
            w = _ptr(seg, "seg", segmented_bytes(N, K))
            xp = _ptr(x, "x", M * K * 2, 2)
            yp = _ptr(y, "y", M * (N // 2 if gate_up else N) * 2, 2)
            arr[i] = StackJob(w.value, None, xp.value, yp.value, N, K, 1 if gate_up else 0)
            self._keep += [seg, x, y]
        nbytes = ctypes.c_size_t(0)
        _check("zq4_stack_plan_bytes", lib.zq4_stack_plan_bytes(ctypes.cast(arr, ctypes.c_void_p), len(jobs), M, ctypes.byref(nbytes)))
        dev = x.device if jobs else None
        self.buffer = torch.empty(nbytes.value, dtype=torch.uint8, device=dev)
        self.plan = StackPlanC()
        _check("zq4_stack_plan_init",
               lib.zq4_stack_plan_init(ctypes.cast(arr, ctypes.c_void_p), len(jobs), M, ctypes.c_void_p(self.buffer.data_ptr()),
                                       nbytes.value, ctypes.byref(self.plan), _stream(stream)))
        self.n_jobs, self.M = len(jobs), M

    def run(self, stream=None):
        _check("zq4_stack_run", lib.zq4_stack_run(ctypes.byref(self.plan), _stream(stream)))

    def set_wait_limit(self, ns):
        """How long (ns) a device-side wait may last before the launch gives
        up (0: the default, 2 s)."""
        _check("zq4_stack_plan_set_wait_limit", lib.zq4_stack_plan_set_wait_limit(ctypes.byref(self.plan), int(ns)))


class StaticStackPlan:
    """A decode-step plan held in the library's fixed device array
    (zq4_stack_plan_init_static): no device memory is allocated for it. One
    per device at a time; jobs as StackPlan."""

    def __init__(self, jobs, M, stream=None):
        arr = (StackJob * len(jobs))()
        self._keep = []
        for i, (seg, x, y, N, K, gate_up) in enumerate(jobs):
            w = _ptr(seg, "seg", segmented_bytes(N, K))
            xp = _ptr(x, "x", M * K * 2, 2)
            yp = _ptr(y, "y", M * (N // 2 if gate_up else N) * 2, 2)
            arr[i] = StackJob(w.value, None, xp.value, yp.value, N, K, 1 if gate_up else 0)
            self._keep += [seg, x, y]
        self.plan = StackPlanC()
        _check("zq4_stack_plan_init_static",
               lib.zq4_stack_plan_init_static(ctypes.cast(arr, ctypes.c_void_p), len(jobs), M,
                                              ctypes.byref(self.plan), _stream(stream)))
        self.n_jobs, self.M = len(jobs), M

    def run(self, stream=None):
        _check("zq4_stack_run", lib.zq4_stack_run(ctypes.byref(self.plan), _stream(stream)))

