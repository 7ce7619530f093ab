"""ctypes binding of libgqadecode.so (argument marshalling only).

Every function here checks dtypes, shapes, devices and contiguity of torch tensors, then passes
``data_ptr()`` values and the current CUDA stream to the C ABI declared in
``include/gqa_decode.h``.  All arithmetic happens in the library's CUDA kernels; there is no
fallback of any kind: importing this module raises if the library has not been built.
"""

from __future__ import annotations

import ctypes
import math
from pathlib import Path

import torch

_LIB_PATH = Path(__file__).resolve().parent / "lib" / "libgqadecode.so"

GQA_OK, GQA_EINVAL, GQA_EWORKSPACE, GQA_EUNSUPPORTED, GQA_ECUDA = range(5)
KIND_F16, KIND_Q8, KIND_TQ = 0, 1, 2
ERR_KVLEN_RANGE, ERR_ID_RANGE, ERR_SEQ_RANGE, ERR_TIMEOUT = 0x1, 0x2, 0x4, 0x8

# Every symbol the header declares (checked by the CPU test suite).
EXPORTS = ("attn_decode_plan", "attn_decode_workspace_bytes", "attn_decode_f16",
           "attn_decode_q8_sel", "attn_merge", "gqa_status_string", "gqa_last_error",
           "gqa_abi_version", "attn_decode_f16_noalloc", "attn_select_topk", "kv_append_q8", "attn_merge_gated",
           "attn_decode_tq", "attn_decode_q8_sel_sg", "kv_append_q8_sg", "attn_decode_f16_gated",
           "attn_decode_q8_sel_gated", "attn_decode_tq_gated")
NOALLOC_SCRATCH_BYTES = 16 << 20  # GQA_NOALLOC_SCRATCH_BYTES in include/gqa_decode.h


class GqaPlan(ctypes.Structure):
    _fields_ = [("chunk", ctypes.c_int), ("n_split", ctypes.c_int), ("tile", ctypes.c_int),
                ("grid_x", ctypes.c_int), ("grid_y", ctypes.c_int), ("grid_z", ctypes.c_int),
                ("merge", ctypes.c_int), ("streamk", ctypes.c_int), ("row_group", ctypes.c_int),
                ("ws_bytes", ctypes.c_size_t)]


class GqaError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"{status}: {msg}")
        self.status = status


def _load():
    if not _LIB_PATH.exists():
        raise ImportError(f"{_LIB_PATH} is missing: build it with "
                          "`python -m gqa_decode_attention_03_gb300.build_lib`")
    lib = ctypes.CDLL(str(_LIB_PATH))
    P, I, I64, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    lib.attn_decode_plan.argtypes = [I, I, I, I, I, I, I, I, I, ctypes.POINTER(GqaPlan)]
    lib.attn_decode_plan.restype = I
    lib.attn_decode_workspace_bytes.argtypes = [I, I, I, I, I, I, I, I]
    lib.attn_decode_workspace_bytes.restype = SZ
    lib.attn_decode_f16.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I64, I, F, P, SZ, P, P]
    lib.attn_decode_f16.restype = I
    lib.attn_decode_q8_sel.argtypes = [P, P, P, P, P, P, I, P, P, P, I, I, I, I, I, I64, I, F, P,
                                       SZ, P, P]
    lib.attn_decode_q8_sel.restype = I
    lib.attn_decode_f16_noalloc.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I64, I, F, P, P]
    lib.attn_decode_f16_noalloc.restype = I
    lib.attn_select_topk.argtypes = [P, I64, P, I, I, I, P, P, P]
    lib.attn_select_topk.restype = I
    lib.kv_append_q8.argtypes = [P, P, I, I, I, P, P, P, P, I, I64, I, I, P]
    lib.kv_append_q8.restype = I
    lib.kv_append_q8_sg.argtypes = [P, P, I, I, I, I, P, P, P, P, I, I64, I, I, P]
    lib.kv_append_q8_sg.restype = I
    lib.attn_decode_q8_sel_sg.argtypes = [P, P, P, P, P, I, P, I, P, P, P, I, I, I, I, I, I64, I,
                                          F, P, SZ, P, P]
    lib.attn_decode_q8_sel_sg.restype = I
    lib.attn_merge_gated.argtypes = [P, P, I, I, I, I, P, I64, P, P]
    lib.attn_merge_gated.restype = I
    lib.attn_decode_tq.argtypes = [P, P, P, P, P, P, P, ctypes.POINTER(F), P, F, F, P, P, P, I,
                                   I, I, I, I, I64, I, P, SZ, P, P]
    lib.attn_decode_tq.restype = I
    lib.attn_decode_f16_gated.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I64, I, F, P, I64, P,
                                          SZ, P, P]
    lib.attn_decode_f16_gated.restype = I
    lib.attn_decode_q8_sel_gated.argtypes = [P, P, P, P, P, I, P, I, P, P, P, I, I, I, I, I, I64,
                                             I, F, P, I64, P, SZ, P, P]
    lib.attn_decode_q8_sel_gated.restype = I
    lib.attn_decode_tq_gated.argtypes = [P, P, P, P, P, P, P, ctypes.POINTER(F), P, F, F, P, P, P,
                                         I, I, I, I, I, I64, I, P, I64, P, SZ, P, P]
    lib.attn_decode_tq_gated.restype = I
    lib.attn_merge.argtypes = [P, P, I, I, I, I, P, P]
    lib.attn_merge.restype = I
    lib.gqa_status_string.argtypes = [I]
    lib.gqa_status_string.restype = ctypes.c_char_p
    lib.gqa_last_error.argtypes = []
    lib.gqa_last_error.restype = ctypes.c_char_p
    lib.gqa_abi_version.argtypes = []
    lib.gqa_abi_version.restype = I
    return lib


LIB = _load()


def _check(status):
    if status != GQA_OK:
        raise GqaError(LIB.gqa_status_string(status).decode(), LIB.gqa_last_error().decode())


def _ptr(x):
    return None if x is None else ctypes.c_void_p(x.data_ptr())


# the current stream's raw handle without building a torch Stream object (several us a call)
_RAW_STREAM = getattr(torch._C, "_cuda_getCurrentRawStream", None)
_GET_DEVICE = getattr(torch._C, "_cuda_getDevice", None)


def _stream(stream):
    if stream is not None:
        return ctypes.c_void_p(stream.cuda_stream)
    if _RAW_STREAM is not None and _GET_DEVICE is not None:
        return ctypes.c_void_p(_RAW_STREAM(_GET_DEVICE()))
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _need(x, dtype, name, ndim=None):
    if not isinstance(x, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if x.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {x.dtype}")
    if not x.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not x.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and x.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {x.dim()}")


def _gate_args(gate, gate_stride, T, H, D):
    """(gate, stride) checked for the gated entry points: fp32 on the device, element (t, h, d)
    at flat index (t*H + h)*stride + d (stride default D; 2*D over [query | gate] pairs)."""
    if gate.dtype != torch.float32 or not gate.is_cuda:
        raise TypeError("gate must be a CUDA fp32 tensor")
    if not gate.is_contiguous():
        raise ValueError("gate must be contiguous")
    gs = D if gate_stride is None else int(gate_stride)
    if gs < D:
        raise ValueError("gate_stride must be >= head_dim")
    if gate.numel() < (T * H - 1) * gs + D:
        raise ValueError("gate too small for its stride")
    return gs


def plan(n_tok, n_heads, n_kv_heads, head_dim, max_kv_len, budget=-1, kind=KIND_F16, num_sms=0,
         n_seq=None):
    """The split plan the decode calls use (host only; num_sms 0 queries the device).
    n_seq: sequences in the cache (default n_tok: every row its own sequence)."""
    p = GqaPlan()
    _check(LIB.attn_decode_plan(n_tok, n_tok if n_seq is None else n_seq, n_heads, n_kv_heads,
                                head_dim, max_kv_len, budget, kind, num_sms, ctypes.byref(p)))
    return p


def workspace_bytes(n_tok, n_heads, n_kv_heads, head_dim, max_kv_len, budget=-1, kind=KIND_F16,
                    n_seq=None):
    return int(LIB.attn_decode_workspace_bytes(n_tok, n_tok if n_seq is None else n_seq, n_heads,
                                               n_kv_heads, head_dim, max_kv_len, budget, kind))


def alloc_workspace(n_tok, n_heads, n_kv_heads, head_dim, max_kv_len, budget=-1, kind=KIND_F16,
                    device=None, n_seq=None):
    """A zeroed workspace: its leading arrival counters must be zero before the first call (every
    call leaves them zero again), so one workspace can be reused across calls and shapes."""
    n = workspace_bytes(n_tok, n_heads, n_kv_heads, head_dim, max_kv_len, budget, kind, n_seq)
    return torch.zeros(max(n, 16), dtype=torch.uint8, device=device or "cuda")


def attn_decode_f16(q, k_cache, v_cache, kv_len, scale=None, seq_of=None, max_kv_len=None,
                    out=None, ws=None, err=None, stream=None, gate=None, gate_stride=None):
    """Decode attention over an f16 cache; returns ``out [T][H][D]`` fp32.

    q [T][H][D] fp32; k_cache, v_cache [n_seq][cap][Hk][D] fp16; kv_len [T] int32 (device);
    seq_of [T] int32 or None; max_kv_len: host bound of kv_len (default: the cache capacity).
    gate: optional fp32 sigmoid output gate (attn_decode_f16_gated), see ``_gate_args``.
    """
    _need(q, torch.float32, "q", 3)
    _need(k_cache, torch.float16, "k_cache", 4)
    _need(v_cache, torch.float16, "v_cache", 4)
    _need(kv_len, torch.int32, "kv_len", 1)
    if seq_of is not None:
        _need(seq_of, torch.int32, "seq_of", 1)
    if k_cache.shape != v_cache.shape:
        raise ValueError("k_cache and v_cache shapes differ")
    T, H, D = q.shape
    n_seq, cap, Hk, Dk = k_cache.shape
    if Dk != D or kv_len.numel() != T:
        raise ValueError("shape mismatch between q, caches and kv_len")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    max_kv_len = cap if max_kv_len is None else int(max_kv_len)
    if out is None:
        out = torch.empty_like(q)
    _need(out, torch.float32, "out", 3)
    if ws is None:
        ws = alloc_workspace(T, H, Hk, D, min(max_kv_len, cap), -1, KIND_F16, q.device, n_seq)
    if gate is not None:
        gs = _gate_args(gate, gate_stride, T, H, D)
        _check(LIB.attn_decode_f16_gated(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out),
                                         _ptr(kv_len), _ptr(seq_of), T, n_seq, H, Hk, D, cap,
                                         max_kv_len, scale, _ptr(gate), gs, _ptr(ws),
                                         ws.numel() * ws.element_size(), _ptr(err),
                                         _stream(stream)))
        return out
    _check(LIB.attn_decode_f16(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out), _ptr(kv_len),
                               _ptr(seq_of), T, n_seq, H, Hk, D, cap, max_kv_len, scale, _ptr(ws),
                               ws.numel() * ws.element_size(), _ptr(err), _stream(stream)))
    return out


def attn_decode_f16_noalloc(q, k_cache, v_cache, kv_len, scale=None, seq_of=None,
                            max_kv_len=None, out=None, err=None, stream=None):
    """attn_decode_f16 for callers that cannot allocate device memory: the split partials go to
    a static 16 MiB device array inside the library instead of a caller workspace.  Calls that
    overlap on the GPU share that array and race; sizes needing more scratch are refused."""
    _need(q, torch.float32, "q", 3)
    _need(k_cache, torch.float16, "k_cache", 4)
    _need(v_cache, torch.float16, "v_cache", 4)
    _need(kv_len, torch.int32, "kv_len", 1)
    if seq_of is not None:
        _need(seq_of, torch.int32, "seq_of", 1)
    T, H, D = q.shape
    n_seq, cap, Hk, _ = k_cache.shape
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    max_kv_len = cap if max_kv_len is None else int(max_kv_len)
    if out is None:
        out = torch.empty_like(q)
    _need(out, torch.float32, "out", 3)
    _check(LIB.attn_decode_f16_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out),
                                       _ptr(kv_len), _ptr(seq_of), T, n_seq, H, Hk, D, cap,
                                       max_kv_len, scale, _ptr(err), _stream(stream)))
    return out


def attn_decode_tq(q_rot, q_jl, k_polar, k_jl, k_norms, v_polar, v_norms, centroids, signs,
                   qjl_scale, kv_len, scale=None, seq_of=None, max_kv_len=None, out=None, ws=None,
                   err=None, stream=None, gate=None, gate_stride=None):
    """Decode attention over a TurboQuant-compressed cache; returns ``out [T][H][D]`` fp32.

    q_rot, q_jl [T][H][D] fp32 (the rotated and JL-projected query); packed words as int32 bit
    patterns, head-major: k_polar, v_polar [n_seq][Hk][cap][D/16], k_jl [n_seq][Hk][cap][D/32],
    k_norms, v_norms [n_seq][Hk][cap]; centroids: 4 host floats; signs [D] fp32 on the device.
    """
    _need(q_rot, torch.float32, "q_rot", 3)
    _need(q_jl, torch.float32, "q_jl", 3)
    _need(k_polar, torch.int32, "k_polar", 4)
    _need(k_jl, torch.int32, "k_jl", 4)
    _need(k_norms, torch.int32, "k_norms", 3)
    _need(v_polar, torch.int32, "v_polar", 4)
    _need(v_norms, torch.int32, "v_norms", 3)
    _need(signs, torch.float32, "signs", 1)
    _need(kv_len, torch.int32, "kv_len", 1)
    if seq_of is not None:
        _need(seq_of, torch.int32, "seq_of", 1)
    T, H, D = q_rot.shape
    n_seq, Hk, cap, _ = k_polar.shape
    if (q_jl.shape != q_rot.shape or v_polar.shape != k_polar.shape or k_polar.shape[3] != D // 16
            or k_jl.shape != (n_seq, Hk, cap, D // 32) or k_norms.shape != (n_seq, Hk, cap)
            or v_norms.shape != (n_seq, Hk, cap) or signs.numel() != D or kv_len.numel() != T):
        raise ValueError("shape mismatch between the queries, the packed caches and kv_len")
    cents = (ctypes.c_float * 4)(*[float(x) for x in centroids])
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    max_kv_len = cap if max_kv_len is None else int(max_kv_len)
    if out is None:
        out = torch.empty_like(q_rot)
    _need(out, torch.float32, "out", 3)
    if ws is None:
        ws = alloc_workspace(T, H, Hk, D, min(max_kv_len, cap), -1, KIND_TQ, q_rot.device, n_seq)
    if gate is not None:
        gs = _gate_args(gate, gate_stride, T, H, D)
        _check(LIB.attn_decode_tq_gated(_ptr(q_rot), _ptr(q_jl), _ptr(k_polar), _ptr(k_jl),
                                        _ptr(k_norms), _ptr(v_polar), _ptr(v_norms), cents,
                                        _ptr(signs), float(qjl_scale), scale, _ptr(out),
                                        _ptr(kv_len), _ptr(seq_of), T, n_seq, H, Hk, D, cap,
                                        max_kv_len, _ptr(gate), gs, _ptr(ws),
                                        ws.numel() * ws.element_size(), _ptr(err),
                                        _stream(stream)))
        return out
    _check(LIB.attn_decode_tq(_ptr(q_rot), _ptr(q_jl), _ptr(k_polar), _ptr(k_jl), _ptr(k_norms),
                              _ptr(v_polar), _ptr(v_norms), cents, _ptr(signs), float(qjl_scale),
                              scale, _ptr(out), _ptr(kv_len), _ptr(seq_of), T, n_seq, H, Hk, D,
                              cap, max_kv_len, _ptr(ws), ws.numel() * ws.element_size(),
                              _ptr(err), _stream(stream)))
    return out


def attn_decode_q8_sel(q, kq, vq, ksc, vsc, kv_len, ids=None, budget=None, scale=None,
                       seq_of=None, max_kv_len=None, out=None, ws=None, err=None, stream=None,
                       gate=None, gate_stride=None):
    """Decode attention over an int8 cache with per-64-dim f16 scales; optional selected ids.

    kq, vq [n_seq][cap][Hk][D] int8; ksc, vsc [n_seq][cap][Hk][D/G] fp16, one scale per G = 64
    dims, or 32 (FORWARD_MSL's 32-element blocks), read off the shape; ids [T][budget] int32.
    """
    _need(q, torch.float32, "q", 3)
    _need(kq, torch.int8, "kq", 4)
    _need(vq, torch.int8, "vq", 4)
    _need(ksc, torch.float16, "ksc", 4)
    _need(vsc, torch.float16, "vsc", 4)
    _need(kv_len, torch.int32, "kv_len", 1)
    if seq_of is not None:
        _need(seq_of, torch.int32, "seq_of", 1)
    if ids is not None:
        _need(ids, torch.int32, "ids", 2)
        budget = ids.shape[1] if budget is None else int(budget)
        if budget > ids.shape[1]:
            raise ValueError("budget exceeds the id list width")
        if ids.shape[1] != budget:
            raise ValueError("ids must be [n_tok][budget]")
    T, H, D = q.shape
    n_seq, cap, Hk, Dk = kq.shape
    if (Dk != D or kv_len.numel() != T or ksc.shape[:3] != (n_seq, cap, Hk)
            or vsc.shape != ksc.shape or ksc.shape[3] not in (D // 64, D // 32)):
        raise ValueError("shape mismatch between q, caches, scales and kv_len")
    sg = D // ksc.shape[3]
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    max_kv_len = cap if max_kv_len is None else int(max_kv_len)
    b = -1 if ids is None else budget
    if out is None:
        out = torch.empty_like(q)
    _need(out, torch.float32, "out", 3)
    if ws is None:
        ws = alloc_workspace(T, H, Hk, D, min(max_kv_len, cap), b, KIND_Q8, q.device, n_seq)
    if gate is not None:
        gs = _gate_args(gate, gate_stride, T, H, D)
        _check(LIB.attn_decode_q8_sel_gated(_ptr(q), _ptr(kq), _ptr(vq), _ptr(ksc), _ptr(vsc), sg,
                                            _ptr(ids), 0 if ids is None else budget, _ptr(out),
                                            _ptr(kv_len), _ptr(seq_of), T, n_seq, H, Hk, D, cap,
                                            max_kv_len, scale, _ptr(gate), gs, _ptr(ws),
                                            ws.numel() * ws.element_size(), _ptr(err),
                                            _stream(stream)))
        return out
    _check(LIB.attn_decode_q8_sel_sg(_ptr(q), _ptr(kq), _ptr(vq), _ptr(ksc), _ptr(vsc), sg,
                                     _ptr(ids), 0 if ids is None else budget, _ptr(out),
                                     _ptr(kv_len), _ptr(seq_of), T, n_seq, H, Hk, D, cap,
                                     max_kv_len, scale, _ptr(ws), ws.numel() * ws.element_size(),
                                     _ptr(err), _stream(stream)))
    return out


def attn_select_topk(block_scores, kv_len, budget, max_kv_len=None, ids=None, err=None,
                     stream=None):
    """Selected-cell ids [T][budget] from per-row block scores [T][stride] (4 cells a block)."""
    _need(block_scores, torch.float32, "block_scores", 2)
    _need(kv_len, torch.int32, "kv_len", 1)
    T, stride = block_scores.shape
    if kv_len.numel() != T:
        raise ValueError("kv_len must have one entry per row")
    max_kv_len = 4 * (stride - 1) + 3 if max_kv_len is None else int(max_kv_len)
    if ids is None:
        ids = torch.empty((T, budget), dtype=torch.int32, device=block_scores.device)
    _need(ids, torch.int32, "ids", 2)
    _check(LIB.attn_select_topk(_ptr(block_scores), stride, _ptr(kv_len), T, max_kv_len,
                                int(budget), _ptr(ids), _ptr(err), _stream(stream)))
    return ids


def kv_append_q8(k_new, v_new, kq, vq, ksc, vsc, seq, t0, stream=None):
    """Quantise fp32 rows k_new / v_new [n_new][Hk][D] into positions t0.. of sequence `seq` of
    the int8 cache (kq, vq [n_seq][cap][Hk][D] int8; ksc, vsc [n_seq][cap][Hk][D/G] fp16, one
    scale per G = 64 or 32 dims, read off the shape)."""
    _need(k_new, torch.float32, "k_new", 3)
    _need(v_new, torch.float32, "v_new", 3)
    for name, x, dt in (("kq", kq, torch.int8), ("vq", vq, torch.int8),
                        ("ksc", ksc, torch.float16), ("vsc", vsc, torch.float16)):
        _need(x, dt, name, 4)
    n_new, Hk, D = k_new.shape
    n_seq, cap, Hk2, D2 = kq.shape
    if (v_new.shape != k_new.shape or (Hk2, D2) != (Hk, D) or ksc.shape[:3] != (n_seq, cap, Hk)
            or vsc.shape != ksc.shape or ksc.shape[3] not in (D // 64, D // 32)):
        raise ValueError("shape mismatch between new rows and the cache")
    _check(LIB.kv_append_q8_sg(_ptr(k_new), _ptr(v_new), n_new, Hk, D, D // ksc.shape[3],
                               _ptr(kq), _ptr(vq), _ptr(ksc), _ptr(vsc), n_seq, cap, int(seq),
                               int(t0), _stream(stream)))


def attn_merge(part, n_valid, out=None, gate=None, gate_stride=None, stream=None):
    """LSE merge of partials ``part [T][S][H][D+2]`` over the first n_valid[t] chunks; with
    ``gate`` (fp32, element (t, h, d) at flat index (t*H + h)*gate_stride + d), the merged row
    is multiplied by sigmoid(gate) (attn_merge_gated)."""
    _need(part, torch.float32, "part", 4)
    _need(n_valid, torch.int32, "n_valid", 1)
    T, S, H, D2 = part.shape
    D = D2 - 2
    if out is None:
        out = torch.empty((T, H, D), dtype=torch.float32, device=part.device)
    _need(out, torch.float32, "out", 3)
    if gate is None:
        _check(LIB.attn_merge(_ptr(part), _ptr(n_valid), S, T, H, D, _ptr(out), _stream(stream)))
    else:
        if gate.dtype != torch.float32 or not gate.is_cuda:
            raise TypeError("gate must be a CUDA fp32 tensor")
        gs = D if gate_stride is None else int(gate_stride)
        if gate.dim() != 1 and not gate.is_contiguous():
            raise ValueError("gate must be contiguous")
        if gate.numel() < (T * H - 1) * gs + D:
            raise ValueError("gate too small for its stride")
        _check(LIB.attn_merge_gated(_ptr(part), _ptr(n_valid), S, T, H, D, _ptr(gate), gs,
                                    _ptr(out), _stream(stream)))
    return out
