"""ctypes binding of libcsa.so (see include/csa.h) -- argument marshalling only.

Every function here takes torch tensors that already live on the current CUDA
device, turns them into the C ABI's plain pointers and sizes, and calls the
entry point of the same name on torch's current stream.  No step of the
computation runs in Python, and there is no fallback: if libcsa.so is missing
or the GPU is not an sm_103 part, the calls raise.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# CSA_CHECKS=1 in the environment selects the build with internal bounds
# checks (libcsa_checks.so: same entry points, CSA_DEV_CHECK on a failed check)
LIB_PATH = os.path.join(_HERE, "libcsa_checks.so" if os.environ.get("CSA_CHECKS") == "1"
                        else "libcsa.so")

CSA_OK = 0
STATUS_NAMES = {
    0: "CSA_OK", 1: "CSA_ERR_INVALID_ARGUMENT", 2: "CSA_ERR_UNSUPPORTED", 3: "CSA_ERR_CAPACITY",
    4: "CSA_ERR_CUDA", 5: "CSA_ERR_DEVICE_FAULT", 6: "CSA_ERR_TIMEOUT", 7: "CSA_ERR_WORKSPACE",
}
DEV_BAD_INDEX, DEV_MISSING_SWA, DEV_BAD_LAYOUT = 0x01, 0x02, 0x04
DEV_CAPACITY, DEV_BAD_LENGTH, DEV_TIMEOUT = 0x08, 0x10, 0x20
DEV_CHECK = 0x40

EXPORTS = ("csa_status_string", "csa_abi_version", "csa_workspace_size", "csa_indexer_scores",
           "csa_topk", "csa_indexer_topk", "csa_gather_mixed", "csa_sparse_mqa_decode", "csa_decode",
           "csa_hca_workspace_size", "csa_hca_decode", "csa_fp4_quantize_keys",
           "csa_indexer_scores_fp4", "csa_decode_fp4", "csa_shard_workspace_size",
           "csa_shard_candidates", "csa_shard_merge", "csa_shard_attention", "csa_window_attention",
           "csa_shard_combine")
MAX_SHARDS = 8  # csa_shard_merge's limit (include/csa.h)
FP4_ROW = 80  # bytes per MXFP4 key row (include/csa.h)


class CsaError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn}: {STATUS_NAMES.get(code, code)}")
        self.code = code


class csa_layout_t(ctypes.Structure):
    _fields_ = [
        ("num_seqs", ctypes.c_int32), ("num_tokens", ctypes.c_int32),
        ("total_comp_rows", ctypes.c_int64), ("max_comp_rows", ctypes.c_int64),
        ("tok_seq", ctypes.c_void_p), ("tok_pos", ctypes.c_void_p), ("comp_off", ctypes.c_void_p),
        ("swa_kv", ctypes.c_void_p), ("swa_cap", ctypes.c_int32),
        ("swa_first_pos", ctypes.c_void_p),
    ]


class csa_params_t(ctypes.Structure):
    _fields_ = [
        ("n_ih", ctypes.c_int32), ("ihd", ctypes.c_int32), ("hd", ctypes.c_int32),
        ("n_heads", ctypes.c_int32), ("top_k", ctypes.c_int32), ("window", ctypes.c_int32),
        ("ratio", ctypes.c_int32), ("scale", ctypes.c_float),
    ]


_lib = None


def load() -> ctypes.CDLL:
    """Load libcsa.so, or libcsa_checks.so under CSA_CHECKS=1 (built by
    sparse_compressed_kv_gb300.build); raise if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{os.path.basename(LIB_PATH)} not found at {LIB_PATH}: run the "
                           "build (python -m sparse_compressed_kv_gb300.build --all) first")
    lib = ctypes.CDLL(LIB_PATH)
    P = ctypes.c_void_p
    L = ctypes.POINTER(csa_layout_t)
    Pm = ctypes.POINTER(csa_params_t)
    i32, i64, sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    lib.csa_status_string.argtypes = [ctypes.c_int]
    lib.csa_status_string.restype = ctypes.c_char_p
    lib.csa_abi_version.restype = i32
    lib.csa_workspace_size.argtypes = [L, Pm, ctypes.POINTER(sz)]
    lib.csa_indexer_scores.argtypes = [L, Pm, P, P, P, P, i64, P, P]
    lib.csa_topk.argtypes = [L, Pm, P, i64, P, P, P, P, sz, P]
    lib.csa_indexer_topk.argtypes = [L, Pm, P, P, P, P, P, P, P, sz, P]
    lib.csa_gather_mixed.argtypes = [L, Pm, P, P, P, P, P, P, P]
    lib.csa_sparse_mqa_decode.argtypes = [i32, Pm, P, P, P, P, P, P, P, sz, P]
    lib.csa_decode.argtypes = [L, Pm, P, P, P, P, P, P, P, P, P, P, sz, P]
    lib.csa_hca_workspace_size.argtypes = [L, Pm, ctypes.POINTER(sz)]
    lib.csa_hca_decode.argtypes = [L, Pm, P, P, P, P, P, P, sz, P]
    lib.csa_fp4_quantize_keys.argtypes = [i64, P, P, P]
    lib.csa_indexer_scores_fp4.argtypes = [L, Pm, P, P, P, P, i64, P, P]
    lib.csa_decode_fp4.argtypes = [L, Pm, P, P, P, P, P, P, P, P, P, P, sz, P]
    lib.csa_shard_workspace_size.argtypes = [L, Pm, i64, i64, ctypes.POINTER(sz)]
    lib.csa_shard_candidates.argtypes = [L, Pm, i64, i64, P, P, P, P, P, P, P, P, sz, P]
    lib.csa_shard_merge.argtypes = [i32, i32, i32, ctypes.POINTER(i64), P, P, P, P, P, P, P, P, P]
    lib.csa_shard_attention.argtypes = [L, Pm, i64, i64, P, P, P, P, P, P, P, P, sz, P]
    lib.csa_window_attention.argtypes = [L, Pm, P, P, P, P, P, sz, P]
    lib.csa_shard_combine.argtypes = [i32, i32, i32, P, P, P, P, P, P]
    for fn in EXPORTS[2:]:
        getattr(lib, fn).restype = ctypes.c_int
    _lib = lib
    return lib


def _p(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must live on the GPU")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn: str, code: int):
    if code != CSA_OK:
        raise CsaError(fn, code)


def params(n_heads: int, top_k: int, window: int = 128, ratio: int = 4,
           scale: Optional[float] = None, n_ih: int = 64, ihd: int = 128,
           hd: int = 512) -> csa_params_t:
    return csa_params_t(n_ih, ihd, hd, n_heads, top_k, window, ratio,
                        float(scale if scale is not None else hd ** -0.5))


class Layout:
    """Device-side layout arrays plus the host-side sizes of csa_layout_t."""

    def __init__(self, tok_seq, tok_pos, comp_off, swa_kv, swa_first_pos,
                 max_comp_rows: int, total_comp_rows: Optional[int] = None,
                 swa_cap: Optional[int] = None):
        self.tok_seq = tok_seq
        self.tok_pos = tok_pos
        self.comp_off = comp_off
        self.swa_kv = swa_kv
        self.swa_first_pos = swa_first_pos
        self.max_comp_rows = int(max_comp_rows)
        self.total_comp_rows = int(total_comp_rows if total_comp_rows is not None
                                   else max_comp_rows)
        self.swa_cap = int(swa_cap if swa_cap is not None else swa_kv.shape[1])

    def c(self) -> csa_layout_t:
        return csa_layout_t(
            int(self.comp_off.shape[0] - 1), int(self.tok_seq.shape[0]), self.total_comp_rows,
            self.max_comp_rows, _p(self.tok_seq), _p(self.tok_pos), _p(self.comp_off),
            _p(self.swa_kv), self.swa_cap, _p(self.swa_first_pos))


def status_string(code: int) -> str:
    return load().csa_status_string(code).decode()


def abi_version() -> int:
    return int(load().csa_abi_version())


def csa_workspace_size(layout: Layout, prm: csa_params_t) -> int:
    n = ctypes.c_size_t(0)
    lc = layout.c()
    _check("csa_workspace_size", load().csa_workspace_size(ctypes.byref(lc), ctypes.byref(prm),
                                                           ctypes.byref(n)))
    return int(n.value)


def workspace(layout: Layout, prm: csa_params_t, device=None) -> torch.Tensor:
    """A zero-filled workspace of csa_workspace_size bytes (allocated by torch)."""
    return torch.zeros(csa_workspace_size(layout, prm), dtype=torch.uint8,
                       device=device or layout.tok_seq.device)


def csa_indexer_scores(layout: Layout, prm: csa_params_t, q_idx, w_idx, k_idx, scores,
                       dev_status, stream=None):
    lc = layout.c()
    _check("csa_indexer_scores", load().csa_indexer_scores(
        ctypes.byref(lc), ctypes.byref(prm), _p(q_idx), _p(w_idx), _p(k_idx), _p(scores),
        int(scores.shape[1]), _p(dev_status), _stream(stream)))


def csa_topk(layout: Layout, prm: csa_params_t, scores, idx, n_sel, dev_status, ws,
             stream=None):
    lc = layout.c()
    _check("csa_topk", load().csa_topk(
        ctypes.byref(lc), ctypes.byref(prm), _p(scores), int(scores.shape[1]), _p(idx),
        _p(n_sel), _p(dev_status), _p(ws), int(ws.numel()), _stream(stream)))


def csa_indexer_topk(layout: Layout, prm: csa_params_t, q_idx, w_idx, k_idx, idx, n_sel,
                     dev_status, ws, stream=None):
    lc = layout.c()
    _check("csa_indexer_topk", load().csa_indexer_topk(
        ctypes.byref(lc), ctypes.byref(prm), _p(q_idx), _p(w_idx), _p(k_idx), _p(idx), _p(n_sel),
        _p(dev_status), _p(ws), int(ws.numel()), _stream(stream)))


def csa_gather_mixed(layout: Layout, prm: csa_params_t, idx, n_sel, comp_kv, kv_buf, kv_len,
                     dev_status, stream=None):
    lc = layout.c()
    _check("csa_gather_mixed", load().csa_gather_mixed(
        ctypes.byref(lc), ctypes.byref(prm), _p(idx), _p(n_sel), _p(comp_kv), _p(kv_buf),
        _p(kv_len), _p(dev_status), _stream(stream)))


def csa_sparse_mqa_decode(prm: csa_params_t, q, kv_buf, kv_len, out, dev_status, ws,
                          sinks=None, stream=None):
    _check("csa_sparse_mqa_decode", load().csa_sparse_mqa_decode(
        int(q.shape[0]), ctypes.byref(prm), _p(q), _p(kv_buf), _p(kv_len), _p(sinks), _p(out),
        _p(dev_status), _p(ws), int(ws.numel()), _stream(stream)))


def csa_decode(layout: Layout, prm: csa_params_t, q_idx, w_idx, k_idx, comp_kv, q, out,
               dev_status, ws, idx_out=None, sinks=None, stream=None):
    lc = layout.c()
    _check("csa_decode", load().csa_decode(
        ctypes.byref(lc), ctypes.byref(prm), _p(q_idx), _p(w_idx), _p(k_idx), _p(comp_kv), _p(q),
        _p(sinks), _p(out), _p(idx_out), _p(dev_status), _p(ws), int(ws.numel()),
        _stream(stream)))


def csa_hca_workspace_size(layout: Layout, prm: csa_params_t) -> int:
    n = ctypes.c_size_t(0)
    lc = layout.c()
    _check("csa_hca_workspace_size", load().csa_hca_workspace_size(
        ctypes.byref(lc), ctypes.byref(prm), ctypes.byref(n)))
    return int(n.value)


def hca_workspace(layout: Layout, prm: csa_params_t, device=None) -> torch.Tensor:
    return torch.zeros(csa_hca_workspace_size(layout, prm), dtype=torch.uint8,
                       device=device or layout.tok_seq.device)


def csa_hca_decode(layout: Layout, prm: csa_params_t, comp_kv, q, out, dev_status, ws,
                   sinks=None, stream=None):
    lc = layout.c()
    _check("csa_hca_decode", load().csa_hca_decode(
        ctypes.byref(lc), ctypes.byref(prm), _p(comp_kv), _p(q), _p(sinks), _p(out),
        _p(dev_status), _p(ws), int(ws.numel()), _stream(stream)))


def csa_fp4_quantize_keys(k_idx, k_fp4, stream=None):
    """bf16 keys [R, 128] -> MXFP4 rows [R, 80] uint8 (both on the GPU)."""
    _check("csa_fp4_quantize_keys", load().csa_fp4_quantize_keys(
        int(k_idx.shape[0]), _p(k_idx), _p(k_fp4), _stream(stream)))


def csa_indexer_scores_fp4(layout: Layout, prm: csa_params_t, q_idx, w_idx, k_fp4, scores,
                           dev_status, stream=None):
    lc = layout.c()
    _check("csa_indexer_scores_fp4", load().csa_indexer_scores_fp4(
        ctypes.byref(lc), ctypes.byref(prm), _p(q_idx), _p(w_idx), _p(k_fp4), _p(scores),
        int(scores.shape[1]), _p(dev_status), _stream(stream)))


def csa_decode_fp4(layout: Layout, prm: csa_params_t, q_idx, w_idx, k_fp4, comp_kv, q, out,
                   dev_status, ws, idx_out=None, sinks=None, stream=None):
    lc = layout.c()
    _check("csa_decode_fp4", load().csa_decode_fp4(
        ctypes.byref(lc), ctypes.byref(prm), _p(q_idx), _p(w_idx), _p(k_fp4), _p(comp_kv), _p(q),
        _p(sinks), _p(out), _p(idx_out), _p(dev_status), _p(ws), int(ws.numel()),
        _stream(stream)))


# ---------------------------------------------------------------- sharded decode

def csa_shard_workspace_size(layout: Layout, prm: csa_params_t, lo: int, hi: int) -> int:
    n = ctypes.c_size_t(0)
    lc = layout.c()
    _check("csa_shard_workspace_size", load().csa_shard_workspace_size(
        ctypes.byref(lc), ctypes.byref(prm), int(lo), int(hi), ctypes.byref(n)))
    return int(n.value)


def csa_shard_candidates(layout: Layout, prm: csa_params_t, lo: int, hi: int, q_idx, w_idx,
                         k_idx_shard, cand_score, cand_idx, n_cand, dev_status, ws, stream=None):
    lc = layout.c()
    _check("csa_shard_candidates", load().csa_shard_candidates(
        ctypes.byref(lc), ctypes.byref(prm), int(lo), int(hi), _p(q_idx), _p(w_idx),
        _p(k_idx_shard), _p(cand_score), _p(cand_idx), _p(n_cand), _p(dev_status), _p(ws),
        int(ws.numel()), _stream(stream)))


def csa_shard_merge(bounds, cand_score, cand_idx, n_cand, idx, n_sel, shard_idx, shard_nsel,
                    dev_status, stream=None):
    """cand_* [G, T, top_k], n_cand [G, T] -> idx [T, top_k], n_sel [T],
    shard_idx [G, T, top_k], shard_nsel [G, T]; bounds: G + 1 ints (host)."""
    G, T, K = (int(x) for x in cand_idx.shape)
    b = (ctypes.c_int64 * (G + 1))(*[int(x) for x in bounds])
    _check("csa_shard_merge", load().csa_shard_merge(
        T, K, G, b, _p(cand_score), _p(cand_idx), _p(n_cand), _p(idx), _p(n_sel), _p(shard_idx),
        _p(shard_nsel), _p(dev_status), _stream(stream)))


def csa_shard_attention(layout: Layout, prm: csa_params_t, lo: int, hi: int, shard_idx,
                        shard_nsel, comp_kv_shard, q, part_o, part_ml, dev_status, ws,
                        stream=None):
    lc = layout.c()
    _check("csa_shard_attention", load().csa_shard_attention(
        ctypes.byref(lc), ctypes.byref(prm), int(lo), int(hi), _p(shard_idx), _p(shard_nsel),
        _p(comp_kv_shard), _p(q), _p(part_o), _p(part_ml), _p(dev_status), _p(ws),
        int(ws.numel()), _stream(stream)))


def csa_window_attention(layout: Layout, prm: csa_params_t, q, part_o, part_ml, dev_status, ws,
                         stream=None):
    lc = layout.c()
    _check("csa_window_attention", load().csa_window_attention(
        ctypes.byref(lc), ctypes.byref(prm), _p(q), _p(part_o), _p(part_ml), _p(dev_status),
        _p(ws), int(ws.numel()), _stream(stream)))


def csa_shard_combine(part_o, part_ml, out, dev_status, sinks=None, stream=None):
    """part_o [P, T, H, 512], part_ml [P, T, H, 2] -> out [T, H, 512]."""
    P, T, H, _ = (int(x) for x in part_o.shape)
    _check("csa_shard_combine", load().csa_shard_combine(
        P, T, H, _p(part_o), _p(part_ml), _p(sinks), _p(out), _p(dev_status), _stream(stream)))
