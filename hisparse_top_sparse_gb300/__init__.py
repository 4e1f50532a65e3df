"""Thin Python binding of libhisparse (the C ABI in include/hisparse.h).

Argument marshalling only: every function checks tensor devices, dtypes,
shapes and contiguity, passes raw pointers and the CUDA stream to the C call
of the same name, and raises ``HisparseError`` on a non-zero status. All
computation runs in the library's CUDA kernels; there is no other path. If
the library is not built, every call raises.

PyTorch provides device memory and streams only.
"""

from __future__ import annotations

import ctypes
import os

import torch

from ._build import LIB as _LIB_PATH, build  # noqa: F401

HS_OK = 0
HS_ERR_INVALID_ARG = -1
HS_ERR_CAPACITY = -2
HS_ERR_INDEX = -3
HS_ERR_CUDA = -4
HS_ERR_TIMEOUT = -5
HS_ERR_UNSUPPORTED = -6
HS_STATUS_INDEX = 1
HS_STATUS_CAPACITY = 2
HS_STATUS_TIMEOUT = 4
HS_LOGITS_F32 = 0
HS_LOGITS_BF16 = 1
LATENT_DIM = 576
VALUE_DIM = 512

EXPORTS = (
    "hs_buffer_create", "hs_buffer_destroy", "hs_request_reset", "hs_get_status",
    "hs_buffer_dump", "hs_buffer_clock", "hs_last_error_string", "hs_resolve_topk",
    "hs_swap_in", "hs_sparse_attn_decode", "hs_verify_finalize", "hs_read_probe", "hs_wait_probe",
    "hs_verify_accept_noalloc", "hs_swap_apply_plan", "hs_backup_pages", "hs_reclaim_resident",
    "hs_sparse_attn_decode_mixed", "hs_backup_rows", "hs_backup_indexer",
    "hs_buffer_set_copy_sms", "hs_swap_in_attn_decode", "hs_step_groups",
    "hs_step_overlap_fits",
)


class HisparseError(RuntimeError):
    def __init__(self, code: int, what: str, msg: str):
        super().__init__(f"{what} failed with status {code}: {msg}")
        self.code = code


class _Desc(ctypes.Structure):
    _fields_ = [
        ("max_reqs", ctypes.c_int32), ("slots_per_req", ctypes.c_int32),
        ("step_slots", ctypes.c_int32), ("max_ctx", ctypes.c_int32),
        ("block_size", ctypes.c_int32), ("hbt_stride", ctypes.c_int32),
        ("hot_kv", ctypes.c_void_p), ("host_pool", ctypes.c_void_p),
        ("host_pool_rows", ctypes.c_int64), ("host_block_table", ctypes.c_void_p),
    ]


_lib = None
_P = ctypes.c_void_p
_I = ctypes.c_int32
_I64 = ctypes.c_int64


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"{_LIB_PATH} is missing: build it with __graft_entry__.build() "
                "(there is no fallback implementation)")
        L = ctypes.CDLL(_LIB_PATH)
        sig = {
            "hs_buffer_create": (_I, [ctypes.POINTER(_Desc), ctypes.POINTER(_P)]),
            "hs_buffer_destroy": (_I, [_P]),
            "hs_request_reset": (_I, [_P, _I, _P]),
            "hs_get_status": (_I, [_P, _P, ctypes.POINTER(ctypes.c_uint32)]),
            "hs_buffer_dump": (_I, [_P, _P, _P, _P, _P]),
            "hs_buffer_clock": (_I64, [_P]),
            "hs_buffer_set_copy_sms": (_I, [_P, _I]),
            "hs_last_error_string": (ctypes.c_char_p, []),
            "hs_resolve_topk": (_I, [_P, _P, _P, _I, _P, _I, _I, _I, _I, _P, _P, _P, _P]),
            "hs_swap_in": (_I, [_P, _P, _P, _P, _P, _I, _I, _P, _P, _P, _P]),
            "hs_sparse_attn_decode": (_I, [_P, _P, _I64, _P, _I, _I, _I, ctypes.c_float,
                                           _P, _P, _P, _P]),
            "hs_sparse_attn_decode_mixed": (_I, [_P, _P, _I64, _P, _I64, _P, _P, _I, _P, _I, _I,
                                                 _I, ctypes.c_float, _P, _P, _P, _P]),
            "hs_swap_in_attn_decode": (_I, [_P, _P, _P, _P, _P, _I, _I, _P, _I, ctypes.c_float,
                                            _I, _P, _P, _P, _P, _P, _P, _P]),
            "hs_step_groups": (_I, [_I, _I, _P, _P]),
            "hs_step_overlap_fits": (_I, [_I, _P]),
            "hs_reclaim_resident": (_I, [_P, _I, _I, _P, _I, _P, _P, _P, _P]),
            "hs_verify_finalize": (_I, [_P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P]),
            "hs_read_probe": (_I, [_P, ctypes.c_size_t, _P, _I, _P]),
            "hs_wait_probe": (_I, [_P, _I64, _P]),
            "hs_verify_accept_noalloc": (_I, [_P, _I, _I, _I, _I, _P, _P, _P, _P]),
            "hs_swap_apply_plan": (_I, [_P, _I, _P, _P, _I64, _I, _P]),
            "hs_backup_rows": (_I, [_I, _P, _P, _P, _P, _I, _I, _I64, _I64, _P, _P]),
            "hs_backup_indexer": (_I, [_I, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I64, _I64, _P,
                                       _P]),
            "hs_backup_pages": (_I, [_I, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I64, _I64, _P, _P]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _check(rc: int, what: str) -> None:
    if rc != HS_OK:
        raise HisparseError(rc, what, lib().hs_last_error_string().decode(errors="replace"))


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t, name, dtype=None, shape=None, allow_none=False, device=True):
    if t is None:
        if allow_none:
            return None
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if device and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr() if t.numel() > 0 else None


# ------------------------------------------------------------------ buffer --

class HsBuffer:
    """Owner of an hs_buffer handle (the per-request hot buffer's metadata).
    The tensors passed in stay owned by the caller and must outlive it."""

    def __init__(self, max_reqs, slots_per_req, step_slots, max_ctx, block_size,
                 hot_kv: torch.Tensor, host_pool: torch.Tensor,
                 host_block_table: torch.Tensor):
        S_tot = slots_per_req + step_slots
        _ptr(hot_kv, "hot_kv", torch.bfloat16, (max_reqs * S_tot, LATENT_DIM))
        if host_pool.dtype != torch.bfloat16 or host_pool.dim() != 2 or \
                host_pool.shape[1] != LATENT_DIM or not host_pool.is_contiguous():
            raise ValueError("host_pool must be a contiguous bf16 [rows][576] tensor")
        if not host_pool.is_cuda and not host_pool.is_pinned():
            raise ValueError("host_pool must be pinned host memory or a CUDA tensor")
        _ptr(host_block_table, "host_block_table", torch.int32)
        if host_block_table.dim() != 2 or host_block_table.shape[0] < max_reqs:
            raise ValueError("host_block_table must be int32 [max_reqs][hbt_stride]")
        d = _Desc(max_reqs, slots_per_req, step_slots, max_ctx, block_size,
                  host_block_table.shape[1], hot_kv.data_ptr(), host_pool.data_ptr(),
                  host_pool.shape[0], host_block_table.data_ptr())
        h = ctypes.c_void_p()
        _check(lib().hs_buffer_create(ctypes.byref(d), ctypes.byref(h)), "hs_buffer_create")
        self.handle = h
        self.max_reqs, self.S, self.n_step = max_reqs, slots_per_req, step_slots
        self.S_tot, self.max_ctx, self.block_size = S_tot, max_ctx, block_size
        self.hot_kv, self.host_pool, self.hbt = hot_kv, host_pool, host_block_table

    def close(self):
        if getattr(self, "handle", None):
            lib().hs_buffer_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def clock(self) -> int:
        return int(lib().hs_buffer_clock(self.handle))

    def dump(self, stream=None):
        """(token_slot [max_reqs][max_ctx], slot_token [max_reqs][S],
        slot_ts [max_reqs][S]) as CPU tensors."""
        ts = torch.empty((self.max_reqs, self.max_ctx), dtype=torch.int32)
        st = torch.empty((self.max_reqs, self.S), dtype=torch.int32)
        tt = torch.empty((self.max_reqs, self.S), dtype=torch.int64)
        _check(lib().hs_buffer_dump(self.handle, _stream(stream), ts.data_ptr(),
                                    st.data_ptr(), tt.data_ptr()), "hs_buffer_dump")
        return ts, st, tt


def hs_buffer_create(**kw) -> HsBuffer:
    return HsBuffer(**kw)


def hs_buffer_destroy(buf: HsBuffer) -> None:
    buf.close()


def hs_request_reset(buf: HsBuffer, req: int, stream=None) -> None:
    _check(lib().hs_request_reset(buf.handle, int(req), _stream(stream)), "hs_request_reset")


def hs_buffer_set_copy_sms(buf: HsBuffer, n_sms: int) -> None:
    _check(lib().hs_buffer_set_copy_sms(buf.handle, int(n_sms)), "hs_buffer_set_copy_sms")


def hs_get_status(buf: HsBuffer, stream=None) -> int:
    v = ctypes.c_uint32(0)
    _check(lib().hs_get_status(buf.handle, _stream(stream), ctypes.byref(v)), "hs_get_status")
    return int(v.value)


# ----------------------------------------------------------------- calls --

def hs_resolve_topk(req_id_per_row, row_causal_len, block_table, topk, block_size: int,
                    phys_block_stride: int, out_idx, out_valid=None, status=None,
                    stream=None) -> None:
    R, K = topk.shape
    _check(lib().hs_resolve_topk(
        _ptr(req_id_per_row, "req_id_per_row", torch.int32, (R,)),
        _ptr(row_causal_len, "row_causal_len", torch.int32, (R,)),
        _ptr(block_table, "block_table", torch.int32), block_table.shape[1],
        _ptr(topk, "topk", torch.int32), R, K, block_size, phys_block_stride,
        _ptr(out_idx, "out_idx", torch.int32, (R, K)),
        _ptr(out_valid, "out_valid", torch.int32, (R,), allow_none=True),
        _ptr(status, "status", torch.int32, (1,), allow_none=True),
        _stream(stream)), "hs_resolve_topk")


def hs_swap_in(buf: HsBuffer, req_id_per_row, row_causal_len, kv_len, topk, out_slot_idx,
               out_valid=None, stats=None, stream=None) -> None:
    R, K = topk.shape
    _check(lib().hs_swap_in(
        buf.handle,
        _ptr(req_id_per_row, "req_id_per_row", torch.int32, (R,)),
        _ptr(row_causal_len, "row_causal_len", torch.int32, (R,)),
        _ptr(kv_len, "kv_len", torch.int32, (buf.max_reqs,)),
        _ptr(topk, "topk", torch.int32), R, K,
        _ptr(out_slot_idx, "out_slot_idx", torch.int32, (R, K)),
        _ptr(out_valid, "out_valid", torch.int32, (R,), allow_none=True),
        _ptr(stats, "stats", torch.int64, (2,), allow_none=True),
        _stream(stream)), "hs_swap_in")


def hs_sparse_attn_decode(q, kv, idx, scale: float, out, lse=None, status=None,
                          stream=None) -> None:
    R, H, D = q.shape
    if D != LATENT_DIM:
        raise ValueError("q must be [R][H][576]")
    K = idx.shape[1]
    _check(lib().hs_sparse_attn_decode(
        _ptr(q, "q", torch.bfloat16), _ptr(kv, "kv", torch.bfloat16), kv.shape[0],
        _ptr(idx, "idx", torch.int32, (R, K)), R, H, K, float(scale),
        _ptr(out, "out", torch.bfloat16, (R, H, VALUE_DIM)),
        _ptr(lse, "lse", torch.float32, (R, H), allow_none=True),
        _ptr(status, "status", torch.int32, (1,), allow_none=True),
        _stream(stream)), "hs_sparse_attn_decode")


def hs_swap_in_attn_decode(buf: HsBuffer, req_id_per_row, row_causal_len, kv_len, topk, q,
                           scale: float, out_slot_idx, out, groups=None, out_valid=None,
                           lse=None, stats=None, stream=None) -> None:
    """hs_swap_in followed by hs_sparse_attn_decode over buf's hot cache, the
    copies of later row groups overlapped with the attention of earlier ones.
    groups: None (the library's split) or the end row of each group."""
    R, K = topk.shape
    Rq, H, D = q.shape
    if D != LATENT_DIM or Rq != R:
        raise ValueError("q must be [R][H][576]")
    ends = None
    if groups is not None:
        groups = [int(x) for x in groups]
        ends = (ctypes.c_int32 * max(1, len(groups)))(*groups)
    _check(lib().hs_swap_in_attn_decode(
        buf.handle,
        _ptr(req_id_per_row, "req_id_per_row", torch.int32, (R,)),
        _ptr(row_causal_len, "row_causal_len", torch.int32, (R,)),
        _ptr(kv_len, "kv_len", torch.int32, (buf.max_reqs,)),
        _ptr(topk, "topk", torch.int32), R, K,
        _ptr(q, "q", torch.bfloat16), H, float(scale),
        len(groups) if groups is not None else 0,
        ctypes.cast(ends, ctypes.c_void_p) if ends is not None else None,
        _ptr(out_slot_idx, "out_slot_idx", torch.int32, (R, K)),
        _ptr(out_valid, "out_valid", torch.int32, (R,), allow_none=True),
        _ptr(out, "out", torch.bfloat16, (R, H, VALUE_DIM)),
        _ptr(lse, "lse", torch.float32, (R, H), allow_none=True),
        _ptr(stats, "stats", torch.int64, (2,), allow_none=True),
        _stream(stream)), "hs_swap_in_attn_decode")


def hs_step_groups(R: int, H: int) -> list:
    """End rows of the groups hs_swap_in_attn_decode picks on the current device."""
    n = ctypes.c_int32(0)
    ends = (ctypes.c_int32 * 8)()
    _check(lib().hs_step_groups(int(R), int(H), ctypes.byref(n), ends), "hs_step_groups")
    return [int(ends[i]) for i in range(n.value)]


def hs_step_overlap_fits(max_reqs: int) -> bool:
    """Whether a copy block of hs_swap_in_attn_decode fits on an SM beside an
    attention CTA on the current device (for a buffer of max_reqs requests)."""
    f = ctypes.c_int32(0)
    _check(lib().hs_step_overlap_fits(int(max_reqs), ctypes.byref(f)), "hs_step_overlap_fits")
    return bool(f.value)


def hs_sparse_attn_decode_mixed(q, kv_resident, kv_hot, row_req, fully_resident, idx,
                                scale: float, out, lse=None, status=None, stream=None) -> None:
    """Row r reads kv_resident while fully_resident[row_req[r]] != 0, else
    kv_hot (row_req None: the flags are indexed by row)."""
    R, H, D = q.shape
    if D != LATENT_DIM:
        raise ValueError("q must be [R][H][576]")
    K = idx.shape[1]
    n_reqs = fully_resident.numel() if fully_resident is not None else 0
    _check(lib().hs_sparse_attn_decode_mixed(
        _ptr(q, "q", torch.bfloat16),
        _ptr(kv_resident, "kv_resident", torch.bfloat16), kv_resident.shape[0],
        _ptr(kv_hot, "kv_hot", torch.bfloat16), kv_hot.shape[0],
        _ptr(row_req, "row_req", torch.int32, (R,), allow_none=True),
        _ptr(fully_resident, "fully_resident", torch.int32, allow_none=True), n_reqs,
        _ptr(idx, "idx", torch.int32, (R, K)), R, H, K, float(scale),
        _ptr(out, "out", torch.bfloat16, (R, H, VALUE_DIM)),
        _ptr(lse, "lse", torch.float32, (R, H), allow_none=True),
        _ptr(status, "status", torch.int32, (1,), allow_none=True),
        _stream(stream)), "hs_sparse_attn_decode_mixed")


def hs_reclaim_resident(block_table, n_blocks, need: int, freed=None, fully_resident=None,
                        n_freed=None, stream=None) -> None:
    """Releases up to `need` resident pages (all but each request's last two,
    scan order) in the device block table."""
    B, stride = block_table.shape
    _check(lib().hs_reclaim_resident(
        _ptr(block_table, "block_table", torch.int32), B, stride,
        _ptr(n_blocks, "n_blocks", torch.int32, (B,)), int(need),
        _ptr(freed, "freed", torch.int32, (int(need),), allow_none=True),
        _ptr(fully_resident, "fully_resident", torch.int32, (B,), allow_none=True),
        _ptr(n_freed, "n_freed", torch.int32, (1,), allow_none=True),
        _stream(stream)), "hs_reclaim_resident")


def hs_verify_finalize(buf: HsBuffer, logits, draft_tokens, step_kv, kv_len, accept_len,
                       next_token, req_ids=None, stream=None) -> None:
    B, d1, V = logits.shape
    d = d1 - 1
    if logits.dtype == torch.float32:
        dt = HS_LOGITS_F32
    elif logits.dtype == torch.bfloat16:
        dt = HS_LOGITS_BF16
    else:
        raise TypeError("logits must be float32 or bfloat16")
    _check(lib().hs_verify_finalize(
        buf.handle, _ptr(logits, "logits"), dt, B, d, V,
        _ptr(draft_tokens, "draft_tokens", torch.int32, (B, d), allow_none=(d == 0)),
        _ptr(step_kv, "step_kv", torch.bfloat16, (B, d1, LATENT_DIM)),
        _ptr(req_ids, "req_ids", torch.int32, (B,), allow_none=True),
        _ptr(kv_len, "kv_len", torch.int32, (buf.max_reqs,)),
        _ptr(accept_len, "accept_len", torch.int32, (B,)),
        _ptr(next_token, "next_token", torch.int32, (B,)),
        _stream(stream)), "hs_verify_finalize")


def hs_verify_accept_noalloc(logits, draft_tokens, accept_len, next_token,
                             stream=None) -> None:
    """Greedy acceptance without any allocation (static scratch in the
    library); see include/hisparse.h."""
    B, d1, V = logits.shape
    d = d1 - 1
    if logits.dtype == torch.float32:
        dt = HS_LOGITS_F32
    elif logits.dtype == torch.bfloat16:
        dt = HS_LOGITS_BF16
    else:
        raise TypeError("logits must be float32 or bfloat16")
    # the static scratch and the stream used are those of the current device
    cur = torch.cuda.current_device()
    for name, t in (("logits", logits), ("draft_tokens", draft_tokens),
                    ("accept_len", accept_len), ("next_token", next_token)):
        if isinstance(t, torch.Tensor) and t.is_cuda and t.device.index != cur:
            raise ValueError(f"{name} is on {t.device}, not on the current device cuda:{cur}")
    _check(lib().hs_verify_accept_noalloc(
        _ptr(logits, "logits"), dt, B, d, V,
        _ptr(draft_tokens, "draft_tokens", torch.int32, (B, d), allow_none=(d == 0)),
        _ptr(accept_len, "accept_len", torch.int32, (B,)),
        _ptr(next_token, "next_token", torch.int32, (B,)),
        _stream(stream)), "hs_verify_accept_noalloc")


def hs_read_probe(src: torch.Tensor, sink: torch.Tensor, blocks: int, stream=None) -> None:
    nbytes = src.numel() * src.element_size()
    if not (src.is_cuda or src.is_pinned()):
        raise ValueError("src must be pinned host memory or a CUDA tensor")
    _check(lib().hs_read_probe(src.data_ptr(), nbytes,
                               _ptr(sink, "sink", torch.int64, (blocks,)), blocks,
                               _stream(stream)), "hs_read_probe")

def hs_wait_probe(status: torch.Tensor, max_cycles: int, stream=None) -> None:
    """One bounded device wait that runs out; sets HS_STATUS_TIMEOUT in status."""
    _check(lib().hs_wait_probe(_ptr(status, "status", torch.int32, (1,)), int(max_cycles),
                               _stream(stream)), "hs_wait_probe")


def _ptr_array(tensors, name, dtype, device):
    """A ctypes array of the tensors' data pointers (checked like _ptr)."""
    arr = (ctypes.c_void_p * len(tensors))()
    for i, t in enumerate(tensors):
        arr[i] = _ptr(t, f"{name}[{i}]", dtype, device=device)
    return arr


def hs_swap_apply_plan(buf: "HsBuffer", hot_kv_layers, host_pool_layers, row_offset: int = 0,
                       stream=None) -> None:
    """Repeat buf's latest swap-in copies for follower caches (one per layer;
    [rows][...] tensors of any dtype, the row size taken from them)."""
    if len(hot_kv_layers) != len(host_pool_layers):
        raise ValueError("one host pool per follower cache")
    n = len(hot_kv_layers)
    row_bytes = _row_bytes(list(hot_kv_layers) + list(host_pool_layers)) if n else 4
    hot = _ptr_array(hot_kv_layers, "hot_kv", None, True)
    pools = _ptr_array(host_pool_layers, "host_pools", None, False)
    _check(lib().hs_swap_apply_plan(buf.handle, n, hot, pools, int(row_offset), row_bytes,
                                    _stream(stream)), "hs_swap_apply_plan")


def _row_bytes(tensors) -> int:
    """Bytes per row (dim 0) shared by all the tensors."""
    rb = tensors[0][0].numel() * tensors[0].element_size()
    for t in tensors:
        if t.dim() < 2 or t[0].numel() * t.element_size() != rb:
            raise ValueError("all caches must be [rows][...] with the same row size")
    return rb


def hs_backup_pages(src_caches, dst_caches, src_blocks, dst_blocks, page_offsets,
                    block_rows: int, blocks_per_kv_block: int, status=None, stream=None) -> None:
    """Copy pages of several layers' device caches ([rows][...] tensors) to
    their host caches; row size from the tensors."""
    if len(src_caches) != len(dst_caches):
        raise ValueError("one host cache per layer")
    n = len(src_caches)
    if n == 0:
        return
    row_bytes = src_caches[0][0].numel() * src_caches[0].element_size()
    for t in list(src_caches) + list(dst_caches):
        if t[0].numel() * t.element_size() != row_bytes:
            raise ValueError("all caches must have the same row size")
    nt = dst_blocks.shape[0]
    src = _ptr_array(src_caches, "src_caches", None, True)
    dst = _ptr_array(dst_caches, "dst_caches", None, False)
    _check(lib().hs_backup_pages(
        n, src, dst, _ptr(src_blocks, "src_blocks", torch.int32, (n, nt)),
        _ptr(dst_blocks, "dst_blocks", torch.int32, (nt,)),
        _ptr(page_offsets, "page_offsets", torch.int32, (nt,)), nt, int(block_rows),
        int(blocks_per_kv_block), int(row_bytes), src_caches[0].shape[0], dst_caches[0].shape[0],
        _ptr(status, "status", torch.int32, (1,), allow_none=True), _stream(stream)),
        "hs_backup_pages")


def hs_backup_rows(src_caches, dst_caches, src_slots, dst_slots, status=None,
                   stream=None) -> None:
    """Row dst_slots[i] of every host cache = row src_slots[i] of its device
    cache ([rows][...] tensors, one row = one token's entry)."""
    if len(src_caches) != len(dst_caches):
        raise ValueError("one host cache per layer")
    n_l = len(src_caches)
    if n_l == 0:
        return
    tb = _row_bytes(list(src_caches) + list(dst_caches))
    n = src_slots.shape[0]
    _check(lib().hs_backup_rows(
        n_l, _ptr_array(src_caches, "src_caches", None, True),
        _ptr_array(dst_caches, "dst_caches", None, False),
        _ptr(src_slots, "src_slots", torch.int32, (n,)),
        _ptr(dst_slots, "dst_slots", torch.int32, (n,)), n, tb, src_caches[0].shape[0],
        dst_caches[0].shape[0], _ptr(status, "status", torch.int32, (1,), allow_none=True),
        _stream(stream)), "hs_backup_rows")


def hs_backup_indexer(src_caches, dst_caches, src_slots, host_slots, positions,
                      storage_block_size: int, compress_ratio: int, status=None,
                      stream=None) -> None:
    """hs_backup_rows into the indexer's compressed host cache: the host row
    comes from the logical host slot and the position."""
    if len(src_caches) != len(dst_caches):
        raise ValueError("one host cache per layer")
    n_l = len(src_caches)
    if n_l == 0:
        return
    tb = _row_bytes(list(src_caches) + list(dst_caches))
    n = src_slots.shape[0]
    _check(lib().hs_backup_indexer(
        n_l, _ptr_array(src_caches, "src_caches", None, True),
        _ptr_array(dst_caches, "dst_caches", None, False),
        _ptr(src_slots, "src_slots", torch.int32, (n,)),
        _ptr(host_slots, "host_slots", torch.int32, (n,)),
        _ptr(positions, "positions", torch.int32, (n,)), n, int(storage_block_size),
        int(compress_ratio), tb, src_caches[0].shape[0], dst_caches[0].shape[0],
        _ptr(status, "status", torch.int32, (1,), allow_none=True), _stream(stream)),
        "hs_backup_indexer")
