"""ctypes binding of libfastar.so: one Python function per C entry point, same name.

Argument marshalling only: tensors become (pointer, strides), the current CUDA
stream is passed through, and a non-zero return code raises FastarError.  All
computation happens in the library's CUDA kernels; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libfastar.so")

F32, BF16 = 0, 1
OK, EINVAL, EUNSUPPORTED, ECAPACITY, EWORKSPACE, ECUDA = 0, -1, -2, -3, -4, -5
DEV_BAD_LEN, DEV_BAD_BUCKET, DEV_BAD_INDEX = 1, 2, 4
OP_MATCH, OP_SORT, OP_SPARSE_ATTN, OP_ANNCA, OP_MATCH_ANN, OP_CROSS_ATTN, OP_MATCH_PQ = 1, 2, 3, 4, 5, 6, 7
MAX_B, MAX_R, MAX_P = 256, 8, 1024

_P = ctypes.c_void_p
_I = ctypes.c_int
_L = ctypes.c_int64
_F = ctypes.c_float
_S = ctypes.c_size_t

# name -> argtypes (restype int unless listed in _RESTYPES)
_SIGS = {
    "fastar_version": [],
    "fastar_kernel_launches": [],
    "fastar_last_cuda_error": [],
    "fastar_status_string": [_I],
    "fastar_workspace_bytes": [_I, _I, _L, _L, _I, _I, _I, _L, _I],
    "fastar_bucket_assign": [_P, _I, _I, _L, _I, _L, _L, _P, _I, _I, _P, _P, _P, _P],
    "fastar_bucket_assign_qk": [_P, _P, _I, _I, _L, _I, _L, _L, _P, _I, _I, _P, _P, _P, _P, _P],
    "fastar_tempcache_match": [_P, _P, _I, _I, _L, _I, _L, _L, _P, _P, _P, _L, _F, _P, _P, _P, _P, _P, _P, _P,
                               _S, _P],
    "fastar_tempcache_match_ann": [_P, _P, _I, _I, _L, _I, _L, _L, _I, _I, _P, _P, _P, _P, _P, _L, _P, _P, _F, _P,
                                   _P, _P, _P, _P, _P, _S, _P],
    "fastar_cache_compact": [_I, _I, _L, _I, _L, _P, _P, _L, _L, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                             _P, _P, _P, _P],
    "fastar_cache_compact_merge": [_I, _I, _L, _I, _L, _P, _P, _L, _L, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                   _P, _P, _P, _P, _P, _P, _P, _P, _P, _P],
    "fastar_cache_compact_sorted": [_I, _I, _L, _I, _L, _P, _P, _L, _L, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                    _P, _P, _P, _P, _I, _P, _P, _P, _P, _P, _P, _I, _P, _P, _P, _P],
    "fastar_bucket_sort": [_P, _I, _L, _I, _I, _P, _P, _P, _P, _P],
    "fastar_pq_encode": [_P, _I, _I, _L, _I, _L, _L, _P, _I, _I, _P, _P],
    "fastar_tempcache_match_pq": [_P, _P, _I, _I, _L, _I, _L, _L, _P, _P, _P, _P, _L, _P, _I, _I, _F, _P, _P, _P,
                                  _P, _P, _P, _S, _P],
    "fastar_pq_gather_codes": [_I, _L, _L, _I, _P, _P, _P, _P, _P, _P, _P, _P],
    "fastar_sparse_attn": [_P, _I, _I, _L, _I, _L, _L, _I, _I, _P, _P, _P, _P, _L, _P, _P, _F, _P, _L, _L, _P, _P,
                           _P, _S, _P],
    "fastar_sparse_attn_grouped": [_P, _I, _I, _L, _I, _L, _L, _I, _I, _P, _P, _P, _P, _L, _P, _P, _P, _F, _P, _L,
                                   _L, _P, _P, _P, _S, _P],
    "fastar_sparse_attn_presorted": [_P, _I, _I, _L, _I, _L, _L, _I, _I, _P, _P, _P, _P, _L, _P, _P, _P, _P, _F,
                                     _P, _L, _L, _P, _P, _P, _S, _P],
    "fastar_annca_select": [_P, _I, _I, _I, _L, _I, _L, _L, _P, _I, _P, _P, _L, _F, _I, _I, _I, _P, _P, _P, _P, _P,
                            _P, _P, _P, _P, _P, _P, _S, _P],
    "fastar_annca_select_noalloc": [_P, _I, _I, _I, _L, _I, _L, _L, _P, _I, _P, _P, _L, _F, _I, _I, _P, _P, _P, _P],
    "fastar_cross_attn_subset": [_P, _I, _I, _I, _L, _I, _L, _L, _P, _P, _L, _P, _P, _F, _P, _L, _L, _P, _P, _S,
                                 _P],
    "fastar_cross_attn_kept": [_P, _I, _I, _I, _L, _I, _L, _L, _P, _P, _L, _P, _F, _P, _L, _L, _P, _P],
    "fastar_dense_attn": [_P, _I, _I, _L, _I, _L, _L, _P, _P, _L, _L, _L, _F, _P, _L, _L, _P, _P],
    "fastar_dense_attn_grouped": [_P, _I, _I, _L, _I, _L, _L, _P, _P, _L, _L, _L, _P, _L, _F, _P, _L, _L, _P, _P],
    "fastar_dense_append": [_I, _I, _L, _I, _P, _P, _L, _L, _P, _P, _L, _L, _P],
    "fastar_gemm": [_P, _L, _P, _L, _P, _P, _L, _P, _P, _P, _L, _I, _L, _L, _L, _I, _P, _P],
    "fastar_layernorm_mod": [_P, _L, _L, _I, _F, _P, _P, _P, _P, _P, _P, _P, _L, _P],
    "fastar_rmsnorm_rope": [_P, _L, _L, _I, _I, _F, _P, _I, _I, _P, _I, _I, _F, _P],
    "fastar_sinusoidal_embedding": [_P, _I, _I, _P, _L, _P],
}
_RESTYPES = {"fastar_status_string": ctypes.c_char_p, "fastar_workspace_bytes": ctypes.c_size_t,
             "fastar_kernel_launches": ctypes.c_longlong, "fastar_last_cuda_error": ctypes.c_char_p}

_lib: Optional[ctypes.CDLL] = None


class FastarError(RuntimeError):
    def __init__(self, name: str, code: int, detail: str | None = None):
        msg = f"{name} returned {code}: {status_string(code)}"
        super().__init__(msg + (f" ({detail})" if detail else ""))
        self.code = code
        self.detail = detail


def open_library(path: str) -> ctypes.CDLL:
    """Opens a libfastar build and declares every symbol; raises if it is missing."""
    if not os.path.exists(path):
        raise FileNotFoundError(f"{path} is missing: build it with `python -m kv_cache_tempcache_gb300.build_lib`")
    lib = ctypes.CDLL(path)
    for name, args in _SIGS.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = _RESTYPES.get(name, ctypes.c_int)
    return lib


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """The process-wide libfastar handle (opened on first use)."""
    global _lib
    if _lib is None:
        _lib = open_library(path)
    return _lib


def symbols():
    return list(_SIGS)


def status_string(code: int) -> str:
    return load().fastar_status_string(int(code)).decode()


def version() -> int:
    return load().fastar_version()


def kernel_launches() -> int:
    return int(load().fastar_kernel_launches())


def workspace_bytes(op, H, n, M=0, d=128, B=1, r=1, P=0, F=0) -> int:
    return int(load().fastar_workspace_bytes(op, H, n, M, d, B, r, P, F))


# ---- marshalling helpers -------------------------------------------------------------------

def dtype_code(t: torch.dtype) -> int:
    if t == torch.float32:
        return F32
    if t == torch.bfloat16:
        return BF16
    raise TypeError(f"unsupported dtype {t}")


def ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    """Device address of a tensor the library addresses as dense (None -> NULL)."""
    if t is None:
        return None
    if not t.is_contiguous() and t.dim() == 3 and t.stride(2) == 1:
        return t.data_ptr()          # a strided token view; strides are passed separately
    if not t.is_contiguous():
        raise ValueError("index/metadata/output buffers must be contiguous")
    return t.data_ptr()


def stream_handle(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def tok_strides(t: torch.Tensor):
    """(head_stride, token_stride) of a [H, N, d] view with a contiguous last dim."""
    if t.dim() != 3 or t.stride(2) != 1:
        raise ValueError("token tensors must be [H, N, d] views with a contiguous last dimension")
    return t.stride(0), t.stride(1)


def _call(name, *args):
    lib = load()
    rc = getattr(lib, name)(*args)
    if rc != OK:
        detail = lib.fastar_last_cuda_error().decode() if rc == ECUDA else None
        raise FastarError(name, rc, detail)


# ---- entry points --------------------------------------------------------------------------

def fastar_bucket_assign(x, centroids, r, ids, scores=None, norms=None, stream=None):
    H, n, d = x.shape
    hs, ts = tok_strides(x)
    _call("fastar_bucket_assign", ptr(x), dtype_code(x.dtype), H, n, d, hs, ts, ptr(centroids),
          centroids.shape[1], r, ptr(ids), ptr(scores), ptr(norms), stream_handle(stream))


def fastar_bucket_assign_qk(q, k_cur, centroids, r, q_ids, k_ids, k_norms=None, stream=None, q_norms=None):
    H, n, d = q.shape
    hs, ts = tok_strides(q)
    if tok_strides(k_cur) != (hs, ts):
        raise ValueError("q and k_cur must share strides")
    _call("fastar_bucket_assign_qk", ptr(q), ptr(k_cur), dtype_code(q.dtype), H, n, d, hs, ts, ptr(centroids),
          centroids.shape[1], r, ptr(q_ids), ptr(k_ids), ptr(k_norms), ptr(q_norms), stream_handle(stream))


def fastar_tempcache_match(q, k_cur, cache_k, cache_knorm, cache_len, tau, top1, s1, s2, evict, dev_status,
                           workspace, stream=None, owner=None):
    H, nq, d = q.shape
    hs, ts = tok_strides(q)
    if tok_strides(k_cur) != (hs, ts):
        raise ValueError("q and k_cur must share strides")
    _call("fastar_tempcache_match", ptr(q), ptr(k_cur), dtype_code(q.dtype), H, nq, d, hs, ts, ptr(cache_k),
          ptr(cache_knorm), ptr(cache_len), cache_k.shape[1], float(tau), ptr(top1), ptr(s1), ptr(s2), ptr(evict),
          ptr(owner), ptr(dev_status), ptr(workspace),
          0 if workspace is None else workspace.numel() * workspace.element_size(), stream_handle(stream))


def fastar_tempcache_match_ann(q, k_cur, r, B, qperm, qoff, cache_k, cache_knorm, cache_len, kperm, koff, tau,
                               top1, s1, evict, dev_status, workspace, stream=None, owner=None):
    H, nq, d = q.shape
    hs, ts = tok_strides(q)
    if tok_strides(k_cur) != (hs, ts):
        raise ValueError("q and k_cur must share strides")
    _call("fastar_tempcache_match_ann", ptr(q), ptr(k_cur), dtype_code(q.dtype), H, nq, d, hs, ts, int(r), int(B),
          ptr(qperm), ptr(qoff), ptr(cache_k), ptr(cache_knorm), ptr(cache_len), cache_k.shape[1], ptr(kperm),
          ptr(koff), float(tau), ptr(top1), ptr(s1), ptr(evict), ptr(owner), ptr(dev_status), ptr(workspace),
          0 if workspace is None else workspace.numel() * workspace.element_size(), stream_handle(stream))


def fastar_cache_compact(k_cur, v_cur, kcur_norm, kcur_bucket, k_in, v_in, knorm_in, kb_in, len_in, evict,
                         k_out, v_out, knorm_out, kb_out, len_out, index_map, dev_status, stream=None):
    H, nq, d = k_cur.shape
    hs, ts = tok_strides(k_cur)
    if tok_strides(v_cur) != (hs, ts):
        raise ValueError("k_cur and v_cur must share strides")
    _call("fastar_cache_compact", dtype_code(k_cur.dtype), H, nq, d, k_in.shape[1], ptr(k_cur), ptr(v_cur), hs,
          ts, ptr(kcur_norm), ptr(kcur_bucket), ptr(k_in), ptr(v_in), ptr(knorm_in), ptr(kb_in), ptr(len_in),
          ptr(evict), ptr(k_out), ptr(v_out), ptr(knorm_out), ptr(kb_out), ptr(len_out), ptr(index_map),
          ptr(dev_status), stream_handle(stream))


def fastar_cache_compact_sorted(k_cur, v_cur, kcur_norm, kcur_bucket, k_in, v_in, knorm_in, kb_in, len_in, evict,
                                k_out, v_out, knorm_out, kb_out, len_out, index_map, B, kperm, koff, kpos, k_sorted,
                                v_sorted, dev_status, stream=None, qb=None, qperm=None, qoff=None):
    """qb [H, nq, r] int32 (optional): also sort the step's (query, slot) pairs by bucket
    into qperm [H, nq*r] and qoff [H, B+1] in the same launch as the key sort."""
    H, nq, d = k_cur.shape
    hs, ts = tok_strides(k_cur)
    if tok_strides(v_cur) != (hs, ts):
        raise ValueError("k_cur and v_cur must share strides")
    _call("fastar_cache_compact_sorted", dtype_code(k_cur.dtype), H, nq, d, k_in.shape[1], ptr(k_cur), ptr(v_cur),
          hs, ts, ptr(kcur_norm), ptr(kcur_bucket), ptr(k_in), ptr(v_in), ptr(knorm_in), ptr(kb_in), ptr(len_in),
          ptr(evict), ptr(k_out), ptr(v_out), ptr(knorm_out), ptr(kb_out), ptr(len_out), ptr(index_map), int(B),
          ptr(kperm), ptr(koff), ptr(kpos), ptr(k_sorted), ptr(v_sorted), ptr(qb),
          int(qb.shape[2]) if qb is not None else 0, ptr(qperm), ptr(qoff), ptr(dev_status), stream_handle(stream))


def fastar_cache_compact_merge(k_cur, v_cur, kcur_norm, kcur_bucket, k_in, v_in, knorm_in, kb_in, g_in, len_in,
                               evict, top1, owner, k_out, v_out, knorm_out, kb_out, g_out, len_out, index_map,
                               dev_status, stream=None):
    H, nq, d = k_cur.shape
    hs, ts = tok_strides(k_cur)
    if tok_strides(v_cur) != (hs, ts):
        raise ValueError("k_cur and v_cur must share strides")
    _call("fastar_cache_compact_merge", dtype_code(k_cur.dtype), H, nq, d, k_in.shape[1], ptr(k_cur), ptr(v_cur),
          hs, ts, ptr(kcur_norm), ptr(kcur_bucket), ptr(k_in), ptr(v_in), ptr(knorm_in), ptr(kb_in), ptr(g_in),
          ptr(len_in), ptr(evict), ptr(top1), ptr(owner), ptr(k_out), ptr(v_out), ptr(knorm_out), ptr(kb_out),
          ptr(g_out), ptr(len_out), ptr(index_map), ptr(dev_status), stream_handle(stream))


def fastar_pq_encode(x, codebooks, codes, stream=None):
    """codebooks [H, m, Kc, d/m]; codes [H, n, m] uint8."""
    H, n, d = x.shape
    hs, ts = tok_strides(x)
    _call("fastar_pq_encode", ptr(x), dtype_code(x.dtype), H, n, d, hs, ts, ptr(codebooks), codebooks.shape[1],
          codebooks.shape[2], ptr(codes), stream_handle(stream))


def fastar_tempcache_match_pq(q, k_cur, cache_k, cache_knorm, cache_codes, cache_len, codebooks, tau, top1, s1,
                              evict, dev_status, workspace, stream=None, owner=None):
    H, nq, d = q.shape
    hs, ts = tok_strides(q)
    if tok_strides(k_cur) != (hs, ts):
        raise ValueError("q and k_cur must share strides")
    _call("fastar_tempcache_match_pq", ptr(q), ptr(k_cur), dtype_code(q.dtype), H, nq, d, hs, ts, ptr(cache_k),
          ptr(cache_knorm), ptr(cache_codes), ptr(cache_len), cache_k.shape[1], ptr(codebooks), codebooks.shape[1],
          codebooks.shape[2], float(tau), ptr(top1), ptr(s1), ptr(evict), ptr(owner), ptr(dev_status),
          ptr(workspace), 0 if workspace is None else workspace.numel() * workspace.element_size(),
          stream_handle(stream))


def fastar_pq_gather_codes(codes_in, len_in, codes_cur, index_map, len_out, codes_out, dev_status=None,
                           stream=None):
    H, M, m = codes_in.shape
    _call("fastar_pq_gather_codes", H, codes_cur.shape[1], M, m, ptr(codes_in), ptr(len_in), ptr(codes_cur),
          ptr(index_map), ptr(len_out), ptr(codes_out), ptr(dev_status), stream_handle(stream))


def fastar_bucket_sort(ids, B, perm, offsets, n_valid=None, dev_status=None, stream=None):
    H, n, r = ids.shape
    _call("fastar_bucket_sort", ptr(ids), H, n, r, B, ptr(n_valid), ptr(perm), ptr(offsets), ptr(dev_status),
          stream_handle(stream))


def fastar_sparse_attn(q, r, B, qperm, qoff, k, v, kperm, koff, scale, out, lse, dev_status, workspace,
                       stream=None):
    H, nq, d = q.shape
    qh, qt = tok_strides(q)
    oh, ot = tok_strides(out)
    _call("fastar_sparse_attn", ptr(q), dtype_code(q.dtype), H, nq, d, qh, qt, r, B, ptr(qperm), ptr(qoff), ptr(k),
          ptr(v), k.shape[1], ptr(kperm), ptr(koff), float(scale), ptr(out), oh, ot, ptr(lse), ptr(dev_status),
          ptr(workspace), 0 if workspace is None else workspace.numel() * workspace.element_size(),
          stream_handle(stream))


def fastar_sparse_attn_presorted(q, r, B, qperm, qoff, k, v, kperm, koff, k_sorted, v_sorted, scale, out, lse,
                                 dev_status, workspace, stream=None):
    H, nq, d = q.shape
    qh, qt = tok_strides(q)
    oh, ot = tok_strides(out)
    _call("fastar_sparse_attn_presorted", ptr(q), dtype_code(q.dtype), H, nq, d, qh, qt, r, B, ptr(qperm),
          ptr(qoff), ptr(k), ptr(v), k.shape[1], ptr(kperm), ptr(koff), ptr(k_sorted), ptr(v_sorted), float(scale),
          ptr(out), oh, ot, ptr(lse), ptr(dev_status), ptr(workspace),
          0 if workspace is None else workspace.numel() * workspace.element_size(), stream_handle(stream))


def fastar_sparse_attn_grouped(q, r, B, qperm, qoff, k, v, kperm, koff, group_count, scale, out, lse, dev_status,
                               workspace, stream=None):
    H, nq, d = q.shape
    qh, qt = tok_strides(q)
    oh, ot = tok_strides(out)
    _call("fastar_sparse_attn_grouped", ptr(q), dtype_code(q.dtype), H, nq, d, qh, qt, r, B, ptr(qperm), ptr(qoff),
          ptr(k), ptr(v), k.shape[1], ptr(kperm), ptr(koff), ptr(group_count), float(scale), ptr(out), oh, ot,
          ptr(lse), ptr(dev_status), ptr(workspace),
          0 if workspace is None else workspace.numel() * workspace.element_size(), stream_handle(stream))


def fastar_annca_select(q, F, qb, kp, pb, tau_ca, topk, gate, keep, kidx, kcnt, score=None, workspace=None,
                        stream=None, B=0, qperm=None, qoff=None, vp=None, kp_kept=None, vp_kept=None, q_norms=None):
    """kp_kept / vp_kept [H, F, P, d] (optional, with vp): the kept rows copied by the
    ranking launch, fastar_cross_attn_kept's input.  q_norms [H, F * tpf] (optional): the
    queries' norms as fastar_bucket_assign_qk writes them."""
    H, nq, d = q.shape
    qh, qt = tok_strides(q)
    tpf = nq // F
    _call("fastar_annca_select", ptr(q), dtype_code(q.dtype), H, F, tpf, d, qh, qt, ptr(qb), qb.shape[2], ptr(kp),
          ptr(pb), kp.shape[1], float(tau_ca), int(topk), int(gate), int(B), ptr(qperm), ptr(qoff), ptr(q_norms),
          ptr(keep),
          ptr(kidx), ptr(kcnt), ptr(score), ptr(vp), ptr(kp_kept), ptr(vp_kept),
          ptr(workspace), 0 if workspace is None else workspace.numel() * workspace.element_size(),
          stream_handle(stream))


def fastar_annca_select_noalloc(q, F, qb, kp, pb, tau_ca, topk, gate, keep, kidx, kcnt, stream=None):
    """fastar_annca_select for callers that cannot allocate: the scores go to the
    library's fixed scratch array (no workspace, no score output)."""
    H, nq, d = q.shape
    qh, qt = tok_strides(q)
    tpf = nq // F
    _call("fastar_annca_select_noalloc", ptr(q), dtype_code(q.dtype), H, F, tpf, d, qh, qt, ptr(qb), qb.shape[2],
          ptr(kp), ptr(pb), kp.shape[1], float(tau_ca), int(topk), int(gate), ptr(keep), ptr(kidx), ptr(kcnt),
          stream_handle(stream))


def fastar_cross_attn_subset(q, F, kp, vp, kidx, kcnt, scale, out, lse=None, stream=None, workspace=None):
    H, nq, d = q.shape
    qh, qt = tok_strides(q)
    oh, ot = tok_strides(out)
    _call("fastar_cross_attn_subset", ptr(q), dtype_code(q.dtype), H, F, nq // F, d, qh, qt, ptr(kp), ptr(vp),
          kp.shape[1], ptr(kidx), ptr(kcnt), float(scale), ptr(out), oh, ot, ptr(lse), ptr(workspace),
          0 if workspace is None else workspace.numel() * workspace.element_size(), stream_handle(stream))


def fastar_cross_attn_kept(q, F, kp_kept, vp_kept, kcnt, scale, out, lse=None, stream=None):
    """Cross-attention over the kept-row planes [H, F, P, d] fastar_annca_select wrote."""
    H, nq, d = q.shape
    qh, qt = tok_strides(q)
    oh, ot = tok_strides(out)
    _call("fastar_cross_attn_kept", ptr(q), dtype_code(q.dtype), H, F, nq // F, d, qh, qt, ptr(kp_kept),
          ptr(vp_kept), kp_kept.shape[2], ptr(kcnt), float(scale), ptr(out), oh, ot, ptr(lse), stream_handle(stream))


def fastar_dense_attn(q, k, v, nk, scale, out, lse=None, stream=None):
    H, nq, d = q.shape
    qh, qt = tok_strides(q)
    kh, kt = tok_strides(k)
    oh, ot = tok_strides(out)
    _call("fastar_dense_attn", ptr(q), dtype_code(q.dtype), H, nq, d, qh, qt, ptr(k), ptr(v), int(nk), kh, kt,
          float(scale), ptr(out), oh, ot, ptr(lse), stream_handle(stream))


def fastar_dense_attn_grouped(q, k, v, nk, group_count, scale, out, lse=None, stream=None):
    """group_count: [H, >= nk] int32 (row stride = its second dimension)."""
    H, nq, d = q.shape
    qh, qt = tok_strides(q)
    kh, kt = tok_strides(k)
    oh, ot = tok_strides(out)
    _call("fastar_dense_attn_grouped", ptr(q), dtype_code(q.dtype), H, nq, d, qh, qt, ptr(k), ptr(v), int(nk), kh,
          kt, ptr(group_count), group_count.shape[1], float(scale), ptr(out), oh, ot, ptr(lse),
          stream_handle(stream))


ACT_NONE, ACT_GELU_TANH, ACT_SILU = 0, 1, 2


def fastar_gemm(A, W, C, bias=None, R=None, gate_a=None, gate_b=None, act=ACT_NONE, dev_status=None, stream=None):
    """C = R + gate * act(A @ W^T + bias); A [M, K], W [N, K], C/R [M, N] (2-D row views)."""
    M, K = A.shape
    N = W.shape[0]
    for t in (A, W, C) + ((R,) if R is not None else ()):
        if t.dim() != 2 or t.stride(1) != 1:
            raise ValueError("GEMM operands must be 2-D row-major views")
    _call("fastar_gemm", A.data_ptr(), A.stride(0), W.data_ptr(), W.stride(0), ptr(bias),
          None if R is None else R.data_ptr(), 0 if R is None else R.stride(0), ptr(gate_a), ptr(gate_b),
          C.data_ptr(), C.stride(0), dtype_code(C.dtype), M, N, K, int(act), ptr(dev_status), stream_handle(stream))


def fastar_layernorm_mod(x, out, eps=1e-6, weight=None, bias=None, shift_a=None, shift_b=None, scale_a=None,
                         scale_b=None, stream=None):
    """out = LN(x) [* weight + bias] * (1 + scale) + shift over the rows of x [n, C]."""
    n, C = x.shape
    _call("fastar_layernorm_mod", x.data_ptr(), x.stride(0), n, C, float(eps), ptr(weight), ptr(bias), ptr(shift_a),
          ptr(shift_b), ptr(scale_a), ptr(scale_b), out.data_ptr(), out.stride(0), stream_handle(stream))


def fastar_rmsnorm_rope(x, d, weight=None, rope=False, t0=0, grid=(1, 1), eps=1e-6, theta=10000.0, stream=None,
                        t0_dev=None):
    """In place on x [n, C]: RMS norm (weight given) then rotary positions (rope); the
    chunk's first frame is t0 + t0_dev[0] (t0_dev: optional device int32)."""
    n, C = x.shape
    _call("fastar_rmsnorm_rope", x.data_ptr(), x.stride(0), n, C, int(d), float(eps), ptr(weight), int(bool(rope)),
          int(t0), ptr(t0_dev), int(grid[0]), int(grid[1]), float(theta), stream_handle(stream))


def fastar_sinusoidal_embedding(t, out, stream=None):
    nb, dim = out.shape
    _call("fastar_sinusoidal_embedding", ptr(t), nb, dim, out.data_ptr(), out.stride(0), stream_handle(stream))


def fastar_dense_append(k_cur, v_cur, k_cache, v_cache, at, stream=None):
    H, nq, d = k_cur.shape
    hs, ts = tok_strides(k_cur)
    _call("fastar_dense_append", dtype_code(k_cur.dtype), H, nq, d, ptr(k_cur), ptr(v_cur), hs, ts, ptr(k_cache),
          ptr(v_cache), k_cache.shape[1], int(at), stream_handle(stream))
