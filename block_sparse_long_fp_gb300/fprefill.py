"""ctypes binding of libfprefill (include/fprefill.h).

Argument marshalling only: tensors become device pointers, the varlen
descriptors stay host int32 arrays, and every computation runs in the CUDA
library.  PyTorch provides device memory and the current stream.  There is
no fallback: if the shared library has not been built, loading fails.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, Structure, c_float, c_int, c_longlong, c_size_t, c_uint64, c_void_p

import numpy as np

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build", "libfprefill.so")

FP_OK, FP_ERR_INVALID, FP_ERR_UNSUPPORTED, FP_ERR_WORKSPACE, FP_ERR_CUDA, FP_ERR_DEVICE_BOUNDS, \
    FP_ERR_TIMEOUT = range(7)
FP_BF16, FP_E4M3 = 0, 1
FP_MAX_BATCH = 128
FP_SELECT_THRESHOLD, FP_SELECT_TOPK, FP_SELECT_TOPP = 0, 1, 2
FP_SCORE_PACKED, FP_SCORE_HEAD_UNION = 0, 1
FP_V_TOKEN_MAJOR, FP_V_DIM_MAJOR = 0, 1


class FpParams(Structure):
    _fields_ = [("block", c_int), ("sink_tokens", c_int), ("local_tokens", c_int),
                ("alpha", c_float), ("softmax_scale", c_float), ("mean_correction", c_int),
                ("kv_splits", c_int), ("select_rule", c_int), ("top_k", c_int), ("top_p", c_float),
                ("score_mode", c_int), ("p_terms", c_int)]


class FpProblem(Structure):
    _fields_ = [("batch", c_int), ("h_q", c_int), ("h_kv", c_int), ("d", c_int), ("dtype", c_int),
                ("cu_seqlens_q", c_void_p), ("seqlens_k", c_void_p), ("q_start_pos", c_void_p),
                ("q", c_void_p), ("q_stride_tok", c_longlong), ("q_stride_head", c_longlong),
                ("k_cache", c_void_p), ("v_cache", c_void_p), ("page_size", c_int),
                ("num_pages", c_int), ("block_table", c_void_p), ("max_pages_per_seq", c_int),
                ("q_scale", c_void_p), ("k_scale", c_void_p), ("v_scale", c_void_p), ("v_layout", c_int)]


class FprefillError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} ({status})")
        self.status = status


_lib = None


def lib():
    """The loaded shared library (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"libfprefill is not built ({_LIB_PATH} missing); "
                               "run block_sparse_long_fp_gb300.build.build()")
        L = ctypes.CDLL(_LIB_PATH)
        P, PP = POINTER(FpProblem), POINTER(FpParams)
        sig = {
            "fp_default_params": ([], FpParams),
            "fp_num_rows": ([P, PP], c_longlong),
            "fp_num_key_blocks": ([P, PP], c_longlong),
            "fp_score_size": ([P, PP], c_longlong),
            "fp_total_q": ([P], c_longlong),
            "fp_score_offsets": ([P, PP, c_void_p, c_longlong], c_longlong),
            "fp_discover_workspace_size": ([P, PP], c_size_t),
            "fp_discover": ([P, PP, c_void_p, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p], c_int),
            "fp_select_workspace_size": ([P, PP], c_size_t),
            "fp_select": ([P, PP, c_void_p, c_void_p, c_void_p, c_longlong, c_void_p, c_void_p,
                           c_void_p, c_size_t, c_void_p], c_int),
            "fp_discover_select_workspace_size": ([P, PP], c_size_t),
            "fp_discover_select": ([P, PP, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_longlong, c_void_p,
                                    c_void_p, c_size_t, c_void_p], c_int),
            "fp_attn_workspace_size": ([P, PP], c_size_t),
            "fp_attn_kv_splits": ([P, PP], c_int),
            "fp_sparse_attn": ([P, PP, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                c_void_p, c_size_t, c_void_p], c_int),
            "fp_dense_attn": ([P, PP, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p], c_int),
            "fp_sparse_attn_noalloc": ([P, PP, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                        c_void_p, c_void_p], c_int),
            "fp_reset_status": ([c_void_p, c_void_p], c_int),
            "fp_device_status": ([c_void_p, c_void_p, POINTER(c_int)], c_int),
            "fp_status_string": ([c_int], ctypes.c_char_p),
            "fp_set_wait_limit_ns": ([c_uint64], None),
            "fp_check_wait_timeout": ([c_void_p, c_uint64, c_void_p], c_int),
        }
        for name, (args, res) in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def status_string(s: int) -> str:
    return lib().fp_status_string(int(s)).decode()


def _check(s: int, what: str):
    if s != FP_OK:
        raise FprefillError(s, what)


def default_params(**over) -> FpParams:
    p = lib().fp_default_params()
    for k, v in over.items():
        setattr(p, k, v)
    return p


def _ptr(t) -> int:
    return 0 if t is None else int(t.data_ptr())


def _stream_handle(stream=None) -> int:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


class Layer:
    """One attention layer's operands: device tensors (q, paged k/v caches,
    block table, FP8 scales) plus the host varlen descriptors.

    q: [total_q, h_q, 128] bf16 (or uint8 e4m3 codes); k_cache:
    [num_pages, page_size, h_kv, 128]; v_cache: the same, or
    [num_pages, h_kv, 128, page_size] with v_layout = FP_V_DIM_MAJOR;
    block_table: int32 [batch, max_pages].
    cu_seqlens_q / seqlens_k / q_start_pos: host int sequences.
    """

    def __init__(self, q, k_cache, v_cache, block_table, cu_seqlens_q, seqlens_k, q_start_pos,
                 h_q: int, h_kv: int, dtype: str = "bf16", q_scale=None, k_scale=None, v_scale=None,
                 params: FpParams | None = None, v_layout: int = 0):
        self.q, self.k_cache, self.v_cache, self.block_table = q, k_cache, v_cache, block_table
        self.q_scale, self.k_scale, self.v_scale = q_scale, k_scale, v_scale
        self.cu = np.ascontiguousarray(cu_seqlens_q, dtype=np.int32)
        self.lk = np.ascontiguousarray(seqlens_k, dtype=np.int32)
        self.start = np.ascontiguousarray(q_start_pos, dtype=np.int32)
        self.h_q, self.h_kv = h_q, h_kv
        self.params = params if params is not None else default_params()
        pr = FpProblem()
        pr.batch = len(self.lk)
        pr.h_q, pr.h_kv, pr.d = h_q, h_kv, int(q.shape[-1])
        pr.dtype = FP_BF16 if dtype == "bf16" else FP_E4M3
        pr.cu_seqlens_q = self.cu.ctypes.data
        pr.seqlens_k = self.lk.ctypes.data
        pr.q_start_pos = self.start.ctypes.data
        pr.q = _ptr(q)
        pr.q_stride_tok = int(q.stride(0))
        pr.q_stride_head = int(q.stride(1))
        pr.k_cache, pr.v_cache = _ptr(k_cache), _ptr(v_cache)
        pr.page_size = int(k_cache.shape[1])
        pr.num_pages = int(k_cache.shape[0])
        pr.block_table = _ptr(block_table)
        pr.max_pages_per_seq = int(block_table.shape[1])
        pr.q_scale, pr.k_scale, pr.v_scale = _ptr(q_scale), _ptr(k_scale), _ptr(v_scale)
        pr.v_layout = int(v_layout)
        self.problem = pr
        L = lib()
        pp, pm = ctypes.byref(pr), ctypes.byref(self.params)
        self.rows = int(L.fp_num_rows(pp, pm))
        if self.rows < 0:
            raise FprefillError(FP_ERR_INVALID, "varlen descriptors")
        self.key_blocks = int(L.fp_num_key_blocks(pp, pm))
        self.score_size = int(L.fp_score_size(pp, pm))
        self.total_q = int(L.fp_total_q(pp))
        self.kv_splits = int(L.fp_attn_kv_splits(pp, pm))   # split-KV parts of the attention calls
        self.ws_bytes = max(int(L.fp_discover_workspace_size(pp, pm)),
                            int(L.fp_select_workspace_size(pp, pm)),
                            int(L.fp_discover_select_workspace_size(pp, pm)),
                            int(L.fp_attn_workspace_size(pp, pm)))
        self._ws = None

    def score_offsets(self) -> np.ndarray:
        """fp_score_offsets: int64 [rows + 1], the start of every score-map row
        and, last, the map's size."""
        offs = np.zeros(self.rows + 1, dtype=np.int64)
        n = lib().fp_score_offsets(*self._refs(), offs.ctypes.data, offs.size)
        if n != offs.size:
            raise FprefillError(FP_ERR_INVALID, "fp_score_offsets")
        return offs

    # -- plumbing -------------------------------------------------------------
    def _refs(self):
        return ctypes.byref(self.problem), ctypes.byref(self.params)

    def workspace(self):
        import torch
        if self._ws is None:
            self._ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=self.q.device)
            _check(lib().fp_reset_status(_ptr(self._ws), _stream_handle()), "fp_reset_status")
        return self._ws

    def reset_status(self):
        _check(lib().fp_reset_status(_ptr(self.workspace()), _stream_handle()), "fp_reset_status")

    def check_wait_timeout(self, limit_ns: int):
        """fp_check_wait_timeout on this layer's workspace."""
        _check(lib().fp_check_wait_timeout(_ptr(self.workspace()), int(limit_ns), _stream_handle()),
               "fp_check_wait_timeout")

    def device_status(self) -> int:
        v = c_int(0)
        _check(lib().fp_device_status(_ptr(self.workspace()), _stream_handle(), ctypes.byref(v)),
               "fp_device_status")
        return v.value

    # -- the four stages ----------------------------------------------------------
    def discover(self, k_mean=None, v_mean=None, score=None):
        import torch
        dev = self.q.device
        shape = (self.key_blocks, self.h_kv, int(self.q.shape[-1]))
        k_mean = k_mean if k_mean is not None else torch.empty(shape, dtype=torch.float32, device=dev)
        v_mean = v_mean if v_mean is not None else torch.empty(shape, dtype=torch.float32, device=dev)
        score = score if score is not None else torch.empty(max(1, self.score_size), dtype=torch.float32,
                                                            device=dev)
        ws = self.workspace()
        _check(lib().fp_discover(*self._refs(), _ptr(k_mean), _ptr(v_mean), _ptr(score), _ptr(ws),
                                 self.ws_bytes, _stream_handle()), "fp_discover")
        return k_mean, v_mean, score

    def select(self, score, row_ptr=None, col_idx=None, nnz=None, dense_mask=None):
        import torch
        dev = self.q.device
        row_ptr = row_ptr if row_ptr is not None else torch.empty(self.rows + 1, dtype=torch.int32, device=dev)
        col_idx = col_idx if col_idx is not None else torch.empty(max(1, self.score_size), dtype=torch.int32,
                                                                  device=dev)
        nnz = nnz if nnz is not None else torch.empty(1, dtype=torch.int32, device=dev)
        ws = self.workspace()
        _check(lib().fp_select(*self._refs(), _ptr(score), _ptr(row_ptr), _ptr(col_idx), col_idx.numel(),
                               _ptr(nnz), _ptr(dense_mask), _ptr(ws), self.ws_bytes, _stream_handle()),
               "fp_select")
        return row_ptr, col_idx, nnz

    def discover_select(self, k_mean=None, v_mean=None, score=None, row_ptr=None, col_idx=None, nnz=None):
        """fp_discover_select: block means and the CSR index in one call (the
        score map only when `score` is given)."""
        import torch
        dev = self.q.device
        shape = (self.key_blocks, self.h_kv, int(self.q.shape[-1]))
        k_mean = k_mean if k_mean is not None else torch.empty(shape, dtype=torch.float32, device=dev)
        v_mean = v_mean if v_mean is not None else torch.empty(shape, dtype=torch.float32, device=dev)
        row_ptr = row_ptr if row_ptr is not None else torch.empty(self.rows + 1, dtype=torch.int32, device=dev)
        col_idx = col_idx if col_idx is not None else torch.empty(max(1, self.score_size), dtype=torch.int32,
                                                                  device=dev)
        nnz = nnz if nnz is not None else torch.empty(1, dtype=torch.int32, device=dev)
        ws = self.workspace()
        _check(lib().fp_discover_select(*self._refs(), _ptr(k_mean), _ptr(v_mean), _ptr(score), _ptr(row_ptr),
                                        _ptr(col_idx), col_idx.numel(), _ptr(nnz), _ptr(ws), self.ws_bytes,
                                        _stream_handle()), "fp_discover_select")
        return k_mean, v_mean, row_ptr, col_idx, nnz

    def _out(self, out, lse):
        import torch
        dev = self.q.device
        out = out if out is not None else torch.empty((self.total_q, self.h_q, int(self.q.shape[-1])),
                                                      dtype=torch.bfloat16, device=dev)
        return out, lse

    def sparse_attn(self, row_ptr, col_idx, k_mean, v_mean, out=None, lse=None, want_lse=True):
        import torch
        out, lse = self._out(out, lse)
        if lse is None and want_lse:
            lse = torch.empty((self.h_q, self.total_q), dtype=torch.float32, device=self.q.device)
        ws = self.workspace()
        _check(lib().fp_sparse_attn(*self._refs(), _ptr(row_ptr), _ptr(col_idx), _ptr(k_mean), _ptr(v_mean),
                                    _ptr(out), _ptr(lse), _ptr(ws), self.ws_bytes, _stream_handle()),
               "fp_sparse_attn")
        return out, lse

    def sparse_attn_noalloc(self, row_ptr, col_idx, k_mean, v_mean, out, lse=None, status=None):
        """fp_sparse_attn_noalloc: same result as sparse_attn, with the
        library's built-in scratch instead of a workspace (nothing is
        allocated here either: out, lse and status are the caller's)."""
        _check(lib().fp_sparse_attn_noalloc(*self._refs(), _ptr(row_ptr), _ptr(col_idx), _ptr(k_mean),
                                            _ptr(v_mean), _ptr(out), _ptr(lse), _ptr(status),
                                            _stream_handle()), "fp_sparse_attn_noalloc")
        return out, lse

    def dense_attn(self, out=None, lse=None, want_lse=True):
        import torch
        out, lse = self._out(out, lse)
        if lse is None and want_lse:
            lse = torch.empty((self.h_q, self.total_q), dtype=torch.float32, device=self.q.device)
        ws = self.workspace()
        _check(lib().fp_dense_attn(*self._refs(), _ptr(out), _ptr(lse), _ptr(ws), self.ws_bytes,
                                   _stream_handle()), "fp_dense_attn")
        return out, lse

    def prefill(self, out=None, lse=None, want_lse=False):
        """One pass of the whole path: discover -> select -> sparse attention."""
        k_mean, v_mean, score = self.discover()
        row_ptr, col_idx, nnz = self.select(score)
        out, lse = self.sparse_attn(row_ptr, col_idx, k_mean, v_mean, out=out, lse=lse, want_lse=want_lse)
        return out, lse, (row_ptr, col_idx, nnz)


def layer_from_case(case, device="cuda", params: FpParams | None = None, v_layout: int = 0):
    """Upload a synthetic case (block_sparse_long_fp_gb300.synth.Case) and wrap it.
    v_layout = FP_V_DIM_MAJOR uploads the value cache as [num_pages, h_kv, 128,
    page_size] (the same values, keys contiguous)."""
    import torch
    spec = case.spec
    v_host = case.v_cache if v_layout == FP_V_TOKEN_MAJOR else np.ascontiguousarray(case.v_cache.transpose(0, 2, 3, 1))
    if spec.dtype == "bf16":
        q = torch.from_numpy(case.q).view(torch.bfloat16).to(device)
        k = torch.from_numpy(case.k_cache).view(torch.bfloat16).to(device)
        v = torch.from_numpy(v_host).view(torch.bfloat16).to(device)
        qs = ks = vs = None
    else:
        q = torch.from_numpy(case.q).to(device)
        k = torch.from_numpy(case.k_cache).to(device)
        v = torch.from_numpy(v_host).to(device)
        qs = torch.from_numpy(case.q_scale).to(device)
        ks = torch.from_numpy(case.k_scale).to(device)
        vs = torch.from_numpy(case.v_scale).to(device)
    bt = torch.from_numpy(case.block_table).to(device)
    return Layer(q, k, v, bt, case.cu_seqlens_q, case.seqlens_k, case.q_start_pos, spec.h_q, spec.h_kv,
                 dtype=spec.dtype, q_scale=qs, k_scale=ks, v_scale=vs, params=params, v_layout=v_layout)
