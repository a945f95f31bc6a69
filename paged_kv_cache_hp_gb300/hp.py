"""Thin ctypes binding of libhp.so (include/hp.h): argument marshalling only.

Every function here has the name of the C entry point it calls and returns that
call's integer status (``HP_OK`` = 0); ``status_name`` turns it into the name
``hp_status_string`` gives.  Tensors are torch tensors on the current CUDA
device; their ``data_ptr()`` is passed through unchanged, and ``stream``
defaults to torch's current stream.  Nothing in this module computes any part
of the path: all of it runs in the library's CUDA kernels.  If libhp.so has not
been built, the first call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libhp.so")

HP_OK = 0
DTYPES = {"f32": 0, "f16": 1, "bf16": 2, "i8": 3, "u8": 4, "f64": 5}
IDX_U32, IDX_U64 = 0, 1
PERMISSIVE, HAS_QUANT, HOST_MEMORY, TEST_STALL = 0x1, 0x2, 0x4, 0x100
ATTN_TENSOR_CORES, ATTN_CUDA_CORES = 0x8, 0x10

_lock = threading.Lock()
_lib = None


class HpPagedDesc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint32) for n in
                ("rank", "paged_axis", "has_shard", "flags", "dtype", "index_type")] + \
               [(n, ctypes.c_uint64) for n in
                ("num_pages", "page_size", "num_heads", "head_dim", "num_seqs", "table_len",
                 "scales_len")] + \
               [(n, ctypes.c_void_p) for n in
                ("page_pool", "block_table", "seq_ptr", "seq_lens", "scales")]


class HpQuantDesc(ctypes.Structure):
    _fields_ = [("scheme_tag", ctypes.c_uint32), ("axis", ctypes.c_uint32),
                ("block_size", ctypes.c_uint64), ("count", ctypes.c_uint64),
                ("scales", ctypes.c_void_p), ("zero_points", ctypes.c_void_p)]


PER_TENSOR, PER_CHANNEL, PER_BLOCK_AFFINE = 0x01, 0x02, 0x03


def quant_desc(scheme_tag, scales, zero_points=None, axis=0, block_size=0, count=None):
    """An hp_quant_desc over device tensors (kept alive on the result's `keep`)."""
    q = HpQuantDesc()
    q.scheme_tag, q.axis, q.block_size = scheme_tag, axis, block_size
    q.count = (0 if scales is None else scales.numel()) if count is None else count
    q.scales, q.zero_points = _p(scales), _p(zero_points)
    q.keep = (scales, zero_points)
    return q


def lib():
    """The loaded library; raises RuntimeError when libhp.so is missing."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    "libhp.so is not built (%s); run paged_kv_cache_hp_gb300.build.build()"
                    % LIB_PATH)
            L = ctypes.CDLL(LIB_PATH)
            i, u64, vp = ctypes.c_int, ctypes.c_uint64, ctypes.c_void_p
            D = ctypes.POINTER(HpPagedDesc)
            pu64 = ctypes.POINTER(ctypes.c_uint64)
            sig = {
                "hp_status_string": (ctypes.c_char_p, [i]),
                "hp_workspace_bytes": (i, [D, pu64]),
                "hp_validate": (i, [D, vp, u64, pu64, vp]),
                "hp_plan": (i, [D, u64, vp, u64, vp, vp]),
                "hp_gather": (i, [D, vp, u64, vp, u64, vp, vp]),
                "hp_gather_planned": (i, [D, vp, vp, vp, vp]),
                "hp_gather_dequant": (i, [D, vp, u64, vp, u64, vp, vp]),
                "hp_gather_dequant_planned": (i, [D, vp, vp, vp, vp]),
                "hp_scatter_append": (i, [D, vp, vp, u64, vp, u64, vp, vp]),
                "hp_append_plan": (i, [D, vp, u64, vp, u64, vp, vp]),
                "hp_scatter_append_planned": (i, [D, vp, vp, u64, vp, vp, vp]),
                "hp_validate_append": (i, [D, vp, u64, vp, u64, pu64, vp]),
                "hp_lane_validate": (i, [u64, u64, vp, u64, pu64]),
                "hp_lane_gather": (i, [vp, vp, u64, u64, u64, u64, u64, ctypes.c_uint32, u64,
                                       vp, ctypes.c_uint32, vp, vp]),
                "hp_lane_append": (i, [vp, vp, u64, u64, u64, u64, u64, ctypes.c_uint32, u64,
                                       u64, vp, ctypes.c_uint32, vp, vp]),
                "hp_gather_noalloc": (i, [D, vp, u64, vp, vp]),
                "hp_copy_pages": (i, [vp, u64, u64, ctypes.c_uint32, vp, vp, u64, ctypes.c_uint32,
                                      vp, vp]),
                "hp_attention_decode_workspace_bytes": (i, [D, ctypes.c_uint32, pu64]),
                "hp_attention_decode": (i, [D, vp, vp, ctypes.c_uint32, ctypes.c_float, vp, vp,
                                            u64, vp, vp]),
                "hp_attention_plan": (i, [D, ctypes.c_uint32, vp, u64, vp, vp]),
                "hp_attention_decode_planned": (i, [D, vp, vp, ctypes.c_uint32, ctypes.c_float,
                                                    vp, vp, u64, vp, vp]),
                "hp_from_kernel_layout": (i, [vp, vp, u64, u64, u64, u64, u64, ctypes.c_uint32,
                                              vp]),
                "hp_to_kernel_layout": (i, [vp, vp, u64, u64, u64, u64, u64, ctypes.c_uint32,
                                            vp]),
                "hp_table_workspace_bytes": (i, [u64, pu64]),
                "hp_padded_to_csr": (i, [vp, vp, u64, u64, u64, ctypes.c_uint32, vp, u64, vp, vp,
                                         u64, vp, vp]),
                "hp_csr_to_padded": (i, [vp, u64, vp, u64, u64, u64, ctypes.c_uint32, vp, vp, u64,
                                         vp, vp]),
                "hp_zero_tails_scratch_bytes": (i, [D, pu64]),
                "hp_zero_tails": (i, [D, vp, u64, vp, u64, vp, vp]),
                "hp_gather_dequant_q": (i, [D, ctypes.POINTER(HpQuantDesc), vp, u64, vp, u64, vp,
                                            vp]),
                "hp_gather_dequant_q_planned": (i, [D, ctypes.POINTER(HpQuantDesc), vp, vp, vp,
                                                    vp]),
            }
            for name, (res, args) in sig.items():
                f = getattr(L, name)
                f.restype, f.argtypes = res, args
            _lib = L
    return _lib


def status_name(code: int) -> str:
    return lib().hp_status_string(code).decode()


def _p(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


class PagedDesc:
    """An hp_paged_desc over device tensors, which it keeps alive.

    ``pool`` is any device tensor whose bytes are the page pool; ``table``,
    ``seq_ptr`` and ``lens`` are int32/int64 (or uint32/uint64) device tensors of
    the index type; ``scales`` an fp32 device tensor.  Field overrides (rank,
    has_shard, num_seqs, table_len, ...) exist so that malformed descriptors can
    be expressed.
    """

    def __init__(self, pool, table, seq_ptr, lens, *, num_pages, page_size, num_heads, head_dim,
                 dtype, index_type, scales=None, flags=0, rank=3, paged_axis=0, has_shard=0,
                 num_seqs=None, table_len=None, scales_len=None):
        self._keep = (pool, table, seq_ptr, lens, scales)
        d = HpPagedDesc()
        d.rank, d.paged_axis, d.has_shard, d.flags = rank, paged_axis, has_shard, flags
        d.dtype = DTYPES[dtype] if isinstance(dtype, str) else dtype
        d.index_type = index_type
        d.num_pages, d.page_size, d.num_heads, d.head_dim = num_pages, page_size, num_heads, head_dim
        d.num_seqs = (0 if lens is None else lens.numel()) if num_seqs is None else num_seqs
        d.table_len = (0 if table is None else table.numel()) if table_len is None else table_len
        d.scales_len = (0 if scales is None else scales.numel()) if scales_len is None else scales_len
        d.page_pool, d.block_table, d.seq_ptr = _p(pool), _p(table), _p(seq_ptr)
        d.seq_lens, d.scales = _p(lens), _p(scales)
        self.c = d

    @property
    def ref(self):
        return ctypes.byref(self.c)


def hp_workspace_bytes(desc: PagedDesc):
    n = ctypes.c_uint64(0)
    rc = lib().hp_workspace_bytes(desc.ref, ctypes.byref(n))
    return rc, n.value


def hp_validate(desc, workspace, stream=None):
    """Returns (status, first_bad)."""
    first = ctypes.c_uint64(0)
    rc = lib().hp_validate(desc.ref, _p(workspace), _wsn(workspace), ctypes.byref(first),
                           _stream(stream))
    return rc, first.value


def hp_validate_append(desc, new_ptr, total_new, workspace, stream=None):
    first = ctypes.c_uint64(0)
    rc = lib().hp_validate_append(desc.ref, _p(new_ptr), total_new, _p(workspace),
                                  _wsn(workspace), ctypes.byref(first), _stream(stream))
    return rc, first.value


def _wsn(workspace):
    return 0 if workspace is None else workspace.numel() * workspace.element_size()


def hp_plan(desc, out_tokens, workspace, d_status=None, stream=None):
    return lib().hp_plan(desc.ref, out_tokens, _p(workspace), _wsn(workspace), _p(d_status),
                         _stream(stream))


def hp_gather(desc, out, out_tokens, workspace, d_status=None, stream=None):
    return lib().hp_gather(desc.ref, _p(out), out_tokens, _p(workspace), _wsn(workspace),
                           _p(d_status), _stream(stream))


def hp_gather_planned(desc, out, workspace, d_status=None, stream=None):
    return lib().hp_gather_planned(desc.ref, _p(out), _p(workspace), _p(d_status), _stream(stream))


def hp_gather_dequant(desc, out, out_tokens, workspace, d_status=None, stream=None):
    return lib().hp_gather_dequant(desc.ref, _p(out), out_tokens, _p(workspace), _wsn(workspace),
                                   _p(d_status), _stream(stream))


def hp_gather_dequant_planned(desc, out, workspace, d_status=None, stream=None):
    return lib().hp_gather_dequant_planned(desc.ref, _p(out), _p(workspace), _p(d_status),
                                           _stream(stream))


def hp_scatter_append(desc, new_rows, new_ptr, total_new, workspace, d_status=None, stream=None):
    return lib().hp_scatter_append(desc.ref, _p(new_rows), _p(new_ptr), total_new, _p(workspace),
                                   _wsn(workspace), _p(d_status), _stream(stream))


def hp_append_plan(desc, new_ptr, total_new, workspace, d_status=None, stream=None):
    return lib().hp_append_plan(desc.ref, _p(new_ptr), total_new, _p(workspace), _wsn(workspace),
                                _p(d_status), _stream(stream))


def hp_scatter_append_planned(desc, new_rows, new_ptr, total_new, workspace, d_status=None,
                              stream=None):
    return lib().hp_scatter_append_planned(desc.ref, _p(new_rows), _p(new_ptr), total_new,
                                           _p(workspace), _p(d_status), _stream(stream))


def hp_lane_validate(capacity, page_tokens, table_host):
    """table_host: a contiguous uint64 numpy array (or None).  Returns (status, detail pair)."""
    det = (ctypes.c_uint64 * 2)()
    n = 0 if table_host is None else len(table_host)
    ptr = None if table_host is None or n == 0 else table_host.ctypes.data
    rc = lib().hp_lane_validate(capacity, page_tokens, ptr, n, det)
    return rc, (det[0], det[1])


def hp_lane_gather(pool, table, capacity, page_tokens, batch, kv_heads, width, dtype, n, out,
                   d_status=None, stream=None, flags=0):
    dt = DTYPES[dtype] if isinstance(dtype, str) else dtype
    return lib().hp_lane_gather(_p(pool), _p(table), capacity, page_tokens, batch, kv_heads,
                                width, dt, n, _p(out), flags, _p(d_status), _stream(stream))


def hp_lane_append(pool, table, capacity, page_tokens, batch, kv_heads, width, dtype, n, m,
                   new_rows, d_status=None, stream=None, flags=0):
    dt = DTYPES[dtype] if isinstance(dtype, str) else dtype
    return lib().hp_lane_append(_p(pool), _p(table), capacity, page_tokens, batch, kv_heads,
                                width, dt, n, m, _p(new_rows), flags, _p(d_status),
                                _stream(stream))


def hp_gather_dequant_q(desc, quant, out, out_tokens, workspace, d_status=None, stream=None):
    return lib().hp_gather_dequant_q(desc.ref, None if quant is None else ctypes.byref(quant),
                                     _p(out), out_tokens, _p(workspace), _wsn(workspace),
                                     _p(d_status), _stream(stream))


def hp_gather_dequant_q_planned(desc, quant, out, workspace, d_status=None, stream=None):
    return lib().hp_gather_dequant_q_planned(desc.ref,
                                             None if quant is None else ctypes.byref(quant),
                                             _p(out), _p(workspace), _p(d_status),
                                             _stream(stream))


def hp_copy_pages(pool, num_pages, page_bytes, index_type, src_pages, dst_pages, num_pairs,
                  d_status=None, stream=None, flags=0):
    return lib().hp_copy_pages(_p(pool), num_pages, page_bytes, index_type, _p(src_pages),
                               _p(dst_pages), num_pairs, flags, _p(d_status), _stream(stream))


def hp_zero_tails_scratch_bytes(desc):
    n = ctypes.c_uint64(0)
    rc = lib().hp_zero_tails_scratch_bytes(desc.ref, ctypes.byref(n))
    return rc, n.value


def hp_zero_tails(desc, workspace, scratch, d_status=None, stream=None):
    return lib().hp_zero_tails(desc.ref, _p(workspace), _wsn(workspace), _p(scratch),
                               _wsn(scratch), _p(d_status), _stream(stream))


def hp_attention_decode_workspace_bytes(desc, num_q_heads):
    n = ctypes.c_uint64(0)
    rc = lib().hp_attention_decode_workspace_bytes(desc.ref, num_q_heads, ctypes.byref(n))
    return rc, n.value


def hp_attention_decode(desc, v_pool, q, num_q_heads, scale, out, workspace, d_status=None,
                        stream=None):
    return lib().hp_attention_decode(desc.ref, _p(v_pool), _p(q), num_q_heads, float(scale),
                                     _p(out), _p(workspace), _wsn(workspace), _p(d_status),
                                     _stream(stream))


def hp_attention_plan(desc, num_q_heads, workspace, d_status=None, stream=None):
    return lib().hp_attention_plan(desc.ref, num_q_heads, _p(workspace), _wsn(workspace),
                                   _p(d_status), _stream(stream))


def hp_attention_decode_planned(desc, v_pool, q, num_q_heads, scale, out, workspace,
                                d_status=None, stream=None):
    return lib().hp_attention_decode_planned(desc.ref, _p(v_pool), _p(q), num_q_heads,
                                             float(scale), _p(out), _p(workspace),
                                             _wsn(workspace), _p(d_status), _stream(stream))


def hp_from_kernel_layout(src, dst, num_blocks, block_size, num_heads, head_dim, x, dtype,
                          stream=None):
    dt = DTYPES[dtype] if isinstance(dtype, str) else dtype
    return lib().hp_from_kernel_layout(_p(src), _p(dst), num_blocks, block_size, num_heads,
                                       head_dim, x, dt, _stream(stream))


def hp_to_kernel_layout(src, dst, num_blocks, block_size, num_heads, head_dim, x, dtype,
                        stream=None):
    dt = DTYPES[dtype] if isinstance(dtype, str) else dtype
    return lib().hp_to_kernel_layout(_p(src), _p(dst), num_blocks, block_size, num_heads,
                                     head_dim, x, dt, _stream(stream))


def hp_table_workspace_bytes(batch):
    n = ctypes.c_uint64(0)
    rc = lib().hp_table_workspace_bytes(batch, ctypes.byref(n))
    return rc, n.value


def hp_padded_to_csr(padded, lens, batch, max_blocks, page_size, index_type, table_out,
                     table_cap, seq_ptr_out, workspace, d_status=None, stream=None):
    return lib().hp_padded_to_csr(_p(padded), _p(lens), batch, max_blocks, page_size, index_type,
                                  _p(table_out), table_cap, _p(seq_ptr_out), _p(workspace),
                                  _wsn(workspace), _p(d_status), _stream(stream))


def hp_csr_to_padded(table, table_len, seq_ptr, batch, max_blocks, pad, index_type, padded_out,
                     workspace, d_status=None, stream=None):
    return lib().hp_csr_to_padded(_p(table), table_len, _p(seq_ptr), batch, max_blocks, pad,
                                  index_type, _p(padded_out), _p(workspace), _wsn(workspace),
                                  _p(d_status), _stream(stream))


def hp_gather_noalloc(desc, out, out_tokens, d_status=None, stream=None):
    """hp_gather with the library's built-in scratch instead of a caller workspace, for
    callers that cannot allocate device memory (at most 16384 sequences; calls must not
    overlap on the GPU)."""
    return lib().hp_gather_noalloc(desc.ref, _p(out), out_tokens, _p(d_status), _stream(stream))


def workspace_for(desc: PagedDesc, device="cuda"):
    """A zeroed, 256-byte-aligned uint8 device workspace of hp_workspace_bytes bytes."""
    import torch
    rc, n = hp_workspace_bytes(desc)
    if rc:
        raise RuntimeError(status_name(rc))
    return torch.zeros(max(n, 256), dtype=torch.uint8, device=device)
