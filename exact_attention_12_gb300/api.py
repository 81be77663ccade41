"""Python binding of the C interface: argument marshalling only.

Every step of the computation runs in the CUDA library; this module checks
tensor shapes/devices, fills `attn_params`, allocates outputs and the
workspace with torch, and calls `attn_fwd` / `attn_bwd` on the current
stream.
"""

import ctypes
import math

import torch

from . import _abi
from ._abi import AttnParams, check_status, lib

_DTYPES = {torch.bfloat16: _abi.ATTN_BF16, torch.float32: _abi.ATTN_FP32}
_FP8 = getattr(torch, "float8_e4m3fn", None)
if _FP8 is not None:
    _DTYPES[_FP8] = _abi.ATTN_FP8_E4M3
_workspaces = {}
_retired = {}


def workspace(device, nbytes):
    """A zero-initialised device workspace of at least `nbytes`, cached per device.

    The cached buffer is shared by every call on that device that does not
    pass its own workspace, so calls that overlap on different streams must
    pass separate workspaces.  When a call needs more, the cache grows to at
    least twice its size; the buffer it replaces stays allocated for the life
    of the process, because a CUDA graph captured earlier still holds its
    address.
    """
    dev = torch.device(device)
    key = (dev.type, dev.index)
    t = _workspaces.get(key)
    if t is None or t.numel() < nbytes:
        size = max(int(nbytes), 256, 0 if t is None else 2 * t.numel())
        if t is not None:
            _retired.setdefault(key, []).append(t)
        t = torch.zeros(size, dtype=torch.uint8, device=dev)
        _workspaces[key] = t
    return t


def _stream(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def make_params(q, *, k=None, scale=None, causal=False, key_lens=None, dropout_p=0.0, seed=0,
                offset=0, block_mask=None, q_descale=None, k_descale=None, v_descale=None):
    """Fill `attn_params` from the query tensor, the key tensor (for its head
    count and strides; None = laid out like q) and the options.  The
    de-scale factors apply to E4M3 inputs only (None = 1)."""
    if q.dim() != 4:
        raise ValueError("tensors must be [B, H, N, d]")
    B, H, N, d = q.shape
    if q.dtype not in _DTYPES:
        raise TypeError(f"unsupported dtype {q.dtype}")
    p = AttnParams()
    p.B, p.H, p.N, p.d = B, H, N, d
    p.dtype = _DTYPES[q.dtype]
    p.scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    p.causal = 1 if causal else 0
    p.dropout_p = float(dropout_p)
    p.philox_seed = int(seed) & 0xFFFFFFFFFFFFFFFF
    p.philox_offset = int(offset)
    p.q_descale = 0.0 if q_descale is None else float(q_descale)
    p.k_descale = 0.0 if k_descale is None else float(k_descale)
    p.v_descale = 0.0 if v_descale is None else float(v_descale)
    sb, sh, sn, sd = q.stride()
    if sd != 1 and d > 1:
        raise ValueError("the head dimension must be contiguous")
    p.stride_b, p.stride_h, p.stride_n = sb, sh, sn
    if k is not None:
        if k.dim() != 4 or k.shape[0] != B or k.shape[3] != d:
            raise ValueError("k must be [B, H_kv, N, d] like q")
        if k.stride(3) != 1 and d > 1:
            raise ValueError("the head dimension must be contiguous")
        p.H_kv = k.shape[1]
        p.kv_stride_b, p.kv_stride_h, p.kv_stride_n = k.stride()[:3]
    if key_lens is not None:
        if key_lens.dtype != torch.int32 or key_lens.device != q.device or key_lens.numel() != B:
            raise ValueError("key_lens must be an int32 tensor [B] on the tensors' device")
        p.key_lens = key_lens.data_ptr()
    if block_mask is not None:
        nb = (N + 127) // 128
        if block_mask.dtype != torch.uint8 or block_mask.device != q.device:
            raise ValueError("block_mask must be uint8 on the tensors' device")
        if not block_mask.is_contiguous():
            raise ValueError("block_mask must be contiguous")
        if tuple(block_mask.shape) == (nb, nb):
            p.block_mask_head_stride = 0
        elif tuple(block_mask.shape) == (B, H, nb, nb):
            p.block_mask_head_stride = nb * nb
        else:
            raise ValueError(f"block_mask must be [{nb}, {nb}] or [B, H, {nb}, {nb}]")
        p.block_mask = block_mask.data_ptr()
    return p


def _same_layout(ref, *ts):
    for t in ts:
        if t.shape != ref.shape or t.stride() != ref.stride() or t.device != ref.device \
                or t.dtype != ref.dtype:
            raise ValueError("tensors of one role must share shape, strides, dtype and device")


def _check_kv(q, k, same_n=True):
    if k.device != q.device or k.dtype != q.dtype:
        raise ValueError("k, v must have q's dtype and device")
    H, H_kv = q.shape[1], k.shape[1] if k.dim() == 4 else -1
    divides = H_kv == 0 if H == 0 else (H_kv >= 1 and H % H_kv == 0)
    if k.dim() != 4 or k.shape[0] != q.shape[0] or k.shape[3] != q.shape[3] or not divides \
            or (same_n and k.shape[2] != q.shape[2]):
        raise ValueError("k, v must be [B, H_kv, N, d] with H_kv dividing q's H")


def _like(t):
    return torch.empty_strided(t.shape, t.stride(), dtype=t.dtype, device=t.device)


def workspace_size(params, backward):
    n = lib().attn_workspace_size(ctypes.byref(params), 1 if backward else 0)
    if n == 0:
        check_status(_abi.ATTN_ERR_INVALID_ARG, "attn_workspace_size")
    return n


def attention_fwd(q, k, v, *, scale=None, causal=False, key_lens=None, dropout_p=0.0, seed=0,
                  offset=0, block_mask=None, out=None, lse=None, ws=None, q_descale=None,
                  k_descale=None, v_descale=None):
    """O and the per-row logsumexp L of exact attention (see include/attn.h).

    q: [B, H, N, d]; k, v: [B, H_kv, N, d] with H_kv dividing H (grouped-query
    attention; H_kv = H is multi-head), CUDA tensors (bf16, fp32, or
    float8_e4m3fn with the de-scale factors: the real values are
    descale * tensor); k and v share strides.  Returns (o, lse) with o like q
    (bf16 for E4M3 inputs) and lse fp32 [B, H, N].
    """
    _check_kv(q, k)
    _same_layout(k, v)
    p = make_params(q, k=k, scale=scale, causal=causal, key_lens=key_lens,
                    dropout_p=dropout_p, seed=seed, offset=offset, block_mask=block_mask,
                    q_descale=q_descale, k_descale=k_descale, v_descale=v_descale)
    if _FP8 is not None and q.dtype == _FP8:
        o = torch.empty_strided(q.shape, q.stride(), dtype=torch.bfloat16,
                                device=q.device) if out is None else out
        if o.dtype != torch.bfloat16 or o.shape != q.shape or o.stride() != q.stride() \
                or o.device != q.device:
            raise ValueError("out must be bf16 with q's shape and strides")
    else:
        o = _like(q) if out is None else out
        _same_layout(q, o)
    B, H, N, _ = q.shape
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    w = workspace(q.device, workspace_size(p, False)) if ws is None else ws
    st = lib().attn_fwd(ctypes.byref(p), q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                        lse.data_ptr(), w.data_ptr(), w.numel() * w.element_size(),
                        _stream(q.device))
    check_status(st, "attn_fwd")
    return o, lse


def attention_bwd(dout, q, k, v, o, lse, *, scale=None, causal=False, key_lens=None,
                  dropout_p=0.0, seed=0, offset=0, block_mask=None, dq=None, dk=None, dv=None,
                  ws=None):
    """dQ, dK, dV of exact attention given the forward's o and lse (bf16).

    dq is like q; dk, dv are like k ([B, H_kv, N, d]; a shared key/value
    head's gradient sums over its group of query heads).
    """
    _check_kv(q, k)
    _same_layout(q, o, dout)
    _same_layout(k, v)
    p = make_params(q, k=k, scale=scale, causal=causal, key_lens=key_lens,
                    dropout_p=dropout_p, seed=seed, offset=offset, block_mask=block_mask)
    dq = _like(q) if dq is None else dq
    dk = _like(k) if dk is None else dk
    dv = _like(k) if dv is None else dv
    _same_layout(q, dq)
    _same_layout(k, dk, dv)
    w = workspace(q.device, workspace_size(p, True)) if ws is None else ws
    st = lib().attn_bwd(ctypes.byref(p), q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                        lse.data_ptr(), dout.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                        dv.data_ptr(), w.data_ptr(), w.numel() * w.element_size(),
                        _stream(q.device))
    check_status(st, "attn_bwd")
    return dq, dk, dv


def attention_decode(q, k, v, cache_lens, *, scale=None, causal=True, out=None, lse=None,
                     ws=None):
    """The decode step: the newest n_q query positions of each sequence against
    its key/value cache (see attn_decode in include/attn.h).

    q: [B, H, n_q, d] bf16; k, v: [B, H_kv, N, d] bf16 caches of capacity N
    with H_kv dividing H; cache_lens: int32 [B] on the device, keys cached per
    sequence.  Query row t of sequence b is the token at position
    cache_lens[b] - n_q + t.  Returns (o, lse) with o like q and lse fp32
    [B, H, n_q].
    """
    _check_kv(q, k, same_n=False)
    _same_layout(k, v)
    n_q = q.shape[2]
    p = make_params(q, k=k, scale=scale, causal=causal, key_lens=cache_lens)
    p.N = k.shape[2]
    o = _like(q) if out is None else out
    _same_layout(q, o)
    B, H = q.shape[:2]
    if lse is None:
        lse = torch.empty((B, H, n_q), dtype=torch.float32, device=q.device)
    need = lib().attn_decode_workspace_size(ctypes.byref(p), n_q)
    if need == 0:
        check_status(_abi.ATTN_ERR_INVALID_ARG, "attn_decode_workspace_size")
    w = workspace(q.device, need) if ws is None else ws
    st = lib().attn_decode(ctypes.byref(p), n_q, q.data_ptr(), k.data_ptr(), v.data_ptr(),
                           o.data_ptr(), lse.data_ptr(), w.data_ptr(),
                           w.numel() * w.element_size(), _stream(q.device))
    check_status(st, "attn_decode")
    return o, lse


def check(ws=None, device=None):
    """Synchronise the current stream and raise if a kernel recorded a time-out."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    w = workspace(dev, 256) if ws is None else ws
    st = lib().attn_check(w.data_ptr(), _stream(dev))
    check_status(st, "attn_check")
