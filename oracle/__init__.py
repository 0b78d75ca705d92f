"""CPU oracle for compressed sparse attention (CSA) decode -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The
product path (``sparse_compressed_kv_gb300``) never does, and the two share no
code: the arithmetic lives in ``csa_oracle.c`` (plain C99, double precision,
optional OpenMP), and this module only marshals numpy arrays through ctypes.

bf16 tensors travel as numpy ``uint16`` bit patterns; the C side widens them
exactly to double.  See ``csa_oracle.h`` for the definitions and the pages
each function follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "csa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle_csa.so")
_default = None
_lock = threading.Lock()

OK = 0
EINVAL = -1
EINDEX = -2
ESWA = -3
ESOFTMAX = -4
ENOMEM = -5


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle's C source into a shared library with gcc (OpenMP on)."""
    hdr = os.path.join(_HERE, "csa_oracle.h")
    if not force and os.path.exists(out) and os.path.getmtime(out) >= max(
            os.path.getmtime(src), os.path.getmtime(hdr)):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp", "-Wall", "-Wextra",
           "-I", _HERE, "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _bind(lib):
    i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
    p = ctypes.c_void_p
    lib.csa_oracle_num_threads.restype = i32
    lib.csa_oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
    lib.csa_oracle_bf16_to_f64.restype = f64
    lib.csa_oracle_n_vis.argtypes = [i64, i64, i32]
    lib.csa_oracle_n_vis.restype = i64
    lib.csa_oracle_block_score.argtypes = [i32, i32, p, p, p]
    lib.csa_oracle_block_score.restype = f64
    lib.csa_oracle_indexer_scores.argtypes = [i32, i32, i32, i32, i32, p, p, p, p, p, p, p, i64,
                                              p]
    lib.csa_oracle_indexer_scores.restype = i32
    lib.csa_oracle_topk.argtypes = [i64, p, i32, p, p]
    lib.csa_oracle_topk.restype = i32
    lib.csa_oracle_gather.argtypes = [i32, i32, i32, i32, i32, i32, p, p, p, p, p, p, p, i32, p,
                                      p, p]
    lib.csa_oracle_gather.restype = i32
    lib.csa_oracle_attention.argtypes = [i32, i32, i32, i64, p, p, p, f64, p, p]
    lib.csa_oracle_attention.restype = i32
    lib.csa_oracle_decode.argtypes = [i32, i32, p, p, p, i32, i32, i32, i32, i32, i32, i32, f64,
                                      p, p, p, p, p, i32, p, p, p, p, i64, p, p, p]
    lib.csa_oracle_decode.restype = i32
    lib.csa_oracle_hca_decode.argtypes = [i32, i32, p, p, p, i32, i32, i32, i32, f64, p, p, i32,
                                          p, p, p, p, p]
    lib.csa_oracle_hca_decode.restype = i32
    lib.csa_oracle_e2m1_value.argtypes = [ctypes.c_uint8]
    lib.csa_oracle_e2m1_value.restype = f64
    lib.csa_oracle_fp4_quantize.argtypes = [i64, i32, p, p]
    lib.csa_oracle_fp4_quantize.restype = i32
    lib.csa_oracle_fp4_dequantize.argtypes = [i64, i32, p, p]
    lib.csa_oracle_fp4_dequantize.restype = i32
    return lib


class OracleError(RuntimeError):
    def __init__(self, fn: str, code: int):
        names = {EINVAL: "EINVAL", EINDEX: "EINDEX", ESWA: "ESWA", ESOFTMAX: "ESOFTMAX",
                 ENOMEM: "ENOMEM"}
        super().__init__(f"{fn} returned {names.get(code, code)}")
        self.code = code


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check(fn, code):
    if code != OK:
        raise OracleError(fn, code)


class Oracle:
    """One loaded copy of the oracle library (the default build, or a copy
    compiled from another source file, e.g. with a planted mistake)."""

    def __init__(self, lib_path: str):
        self.path = lib_path
        self._lib = _bind(ctypes.CDLL(lib_path))

    def num_threads(self) -> int:
        return int(self._lib.csa_oracle_num_threads())


    def bf16_bits_to_f64(self, bits: int) -> float:
        return float(self._lib.csa_oracle_bf16_to_f64(int(bits) & 0xFFFF))


    def n_vis(self, n_comp: int, pos: int, ratio: int = 4) -> int:
        return int(self._lib.csa_oracle_n_vis(int(n_comp), int(pos), int(ratio)))


    def block_score(self, q_bits: np.ndarray, w: np.ndarray, k_bits: np.ndarray) -> float:
        """One block's indexer score.  q_bits [n_ih, ihd] uint16, w [n_ih], k_bits [ihd]."""
        q_bits = _c(q_bits, np.uint16)
        w = _c(w, np.float32)
        k_bits = _c(k_bits, np.uint16)
        n_ih, ihd = q_bits.shape
        assert w.shape == (n_ih,) and k_bits.shape == (ihd,)
        return float(self._lib.csa_oracle_block_score(n_ih, ihd, _ptr(q_bits), _ptr(w), _ptr(k_bits)))


    def indexer_scores(self, q_idx, w_idx, k_idx, tok_seq, tok_pos, comp_off, ratio=4, ld=None):
        """Scores [T, ld] (float64; NaN where s >= n_vis) and n_vis [T]."""
        q_idx = _c(q_idx, np.uint16)
        w_idx = _c(w_idx, np.float32)
        k_idx = _c(k_idx, np.uint16)
        tok_seq = _c(tok_seq, np.int32)
        tok_pos = _c(tok_pos, np.int64)
        comp_off = _c(comp_off, np.int64)
        T, n_ih, ihd = q_idx.shape
        num_seqs = comp_off.shape[0] - 1
        if ld is None:
            ld = max(1, int((comp_off[1:] - comp_off[:-1]).max(initial=0)))
        scores = np.full((T, ld), np.nan, dtype=np.float64)
        nv = np.zeros(T, dtype=np.int64)
        _check("indexer_scores", self._lib.csa_oracle_indexer_scores(
            T, n_ih, ihd, ratio, num_seqs, _ptr(tok_seq), _ptr(tok_pos), _ptr(comp_off),
            _ptr(q_idx), _ptr(w_idx), _ptr(k_idx), _ptr(scores), ld, _ptr(nv)))
        return scores, nv


    def topk(self, scores: np.ndarray, top_k: int):
        """idx [top_k] int32 ascending (padded with -1) and n_sel for a 1-D score vector."""
        scores = _c(scores, np.float64)
        idx = np.empty(top_k, dtype=np.int32)
        n_sel = np.zeros(1, dtype=np.int32)
        _check("topk", self._lib.csa_oracle_topk(scores.shape[0], _ptr(scores), top_k, _ptr(idx),
                                               _ptr(n_sel)))
        return idx, int(n_sel[0])


    def gather(self, idx, n_sel, comp_kv, swa_kv, tok_seq, tok_pos, comp_off, swa_first_pos,
               top_k, window=128, ratio=4):
        """kv_buf [T, top_k+window, hd] uint16 and kv_len [T]."""
        idx = _c(idx, np.int32)
        n_sel = _c(n_sel, np.int32)
        comp_kv = _c(comp_kv, np.uint16)
        swa_kv = _c(swa_kv, np.uint16)
        tok_seq = _c(tok_seq, np.int32)
        tok_pos = _c(tok_pos, np.int64)
        comp_off = _c(comp_off, np.int64)
        swa_first_pos = _c(swa_first_pos, np.int64)
        T = tok_seq.shape[0]
        hd = comp_kv.shape[-1]
        B, swa_cap, _ = swa_kv.shape
        kv_buf = np.zeros((T, top_k + window, hd), dtype=np.uint16)
        kv_len = np.zeros(T, dtype=np.int32)
        _check("gather", self._lib.csa_oracle_gather(
            T, hd, top_k, window, ratio, B, _ptr(tok_seq), _ptr(tok_pos), _ptr(comp_off),
            _ptr(idx), _ptr(n_sel), _ptr(comp_kv), _ptr(swa_kv), swa_cap, _ptr(swa_first_pos),
            _ptr(kv_buf), _ptr(kv_len)))
        return kv_buf, kv_len


    def attention(self, q, kv_buf, kv_len, scale, sinks=None):
        """out [T, H, hd] float64 for q [T, H, hd] and kv_buf [T, rows, hd] (uint16 bits)."""
        q = _c(q, np.uint16)
        kv_buf = _c(kv_buf, np.uint16)
        kv_len = _c(kv_len, np.int32)
        sinks = None if sinks is None else _c(sinks, np.float32)
        T, H, hd = q.shape
        rows = kv_buf.shape[1]
        out = np.zeros((T, H, hd), dtype=np.float64)
        _check("attention", self._lib.csa_oracle_attention(
            T, H, hd, rows, _ptr(q), _ptr(kv_buf), _ptr(kv_len), float(scale), _ptr(sinks),
            _ptr(out)))
        return out


    def decode(self, q_idx, w_idx, k_idx, comp_kv, swa_kv, q, tok_seq, tok_pos, comp_off,
               swa_first_pos, top_k, window=128, ratio=4, scale=None, sinks=None,
               return_scores=False):
        """The whole step.  Returns (idx [T, top_k], n_sel [T], out [T, H, hd] f64[, scores])."""
        q_idx = _c(q_idx, np.uint16)
        w_idx = _c(w_idx, np.float32)
        k_idx = _c(k_idx, np.uint16)
        comp_kv = _c(comp_kv, np.uint16)
        swa_kv = _c(swa_kv, np.uint16)
        q = _c(q, np.uint16)
        tok_seq = _c(tok_seq, np.int32)
        tok_pos = _c(tok_pos, np.int64)
        comp_off = _c(comp_off, np.int64)
        swa_first_pos = _c(swa_first_pos, np.int64)
        sinks = None if sinks is None else _c(sinks, np.float32)
        T, n_ih, ihd = q_idx.shape
        _, H, hd = q.shape
        B, swa_cap, _ = swa_kv.shape
        if scale is None:
            scale = 1.0 / np.sqrt(hd)
        ld = max(1, int((comp_off[1:] - comp_off[:-1]).max(initial=0)))
        scores = np.full((T, ld), np.nan, dtype=np.float64) if return_scores else None
        idx = np.empty((T, top_k), dtype=np.int32)
        n_sel = np.zeros(T, dtype=np.int32)
        out = np.zeros((T, H, hd), dtype=np.float64)
        _check("decode", self._lib.csa_oracle_decode(
            T, B, _ptr(tok_seq), _ptr(tok_pos), _ptr(comp_off), n_ih, ihd, hd, H, top_k, window,
            ratio, float(scale), _ptr(q_idx), _ptr(w_idx), _ptr(k_idx), _ptr(comp_kv),
            _ptr(swa_kv), swa_cap, _ptr(swa_first_pos), _ptr(q), _ptr(sinks), _ptr(scores), ld,
            _ptr(idx), _ptr(n_sel), _ptr(out)))
        if return_scores:
            return idx, n_sel, out, scores
        return idx, n_sel, out


def _hca_decode(self, comp_kv, swa_kv, q, tok_seq, tok_pos, comp_off, swa_first_pos,
                window=128, ratio=128, scale=None, sinks=None):
    """HCA step: out [T, H, hd] f64 and kv_len [T] (dense over visible blocks + window)."""
    comp_kv = _c(comp_kv, np.uint16)
    swa_kv = _c(swa_kv, np.uint16)
    q = _c(q, np.uint16)
    tok_seq = _c(tok_seq, np.int32)
    tok_pos = _c(tok_pos, np.int64)
    comp_off = _c(comp_off, np.int64)
    swa_first_pos = _c(swa_first_pos, np.int64)
    sinks = None if sinks is None else _c(sinks, np.float32)
    T, H, hd = q.shape
    B, swa_cap, _ = swa_kv.shape
    if scale is None:
        scale = 1.0 / np.sqrt(hd)
    out = np.zeros((T, H, hd), dtype=np.float64)
    kv_len = np.zeros(T, dtype=np.int32)
    _check("hca_decode", self._lib.csa_oracle_hca_decode(
        T, B, _ptr(tok_seq), _ptr(tok_pos), _ptr(comp_off), hd, H, window, ratio, float(scale),
        _ptr(comp_kv), _ptr(swa_kv), swa_cap, _ptr(swa_first_pos), _ptr(q), _ptr(sinks),
        _ptr(kv_len), _ptr(out)))
    return out, kv_len


Oracle.hca_decode = _hca_decode

FP4_ROW = 80  # bytes per MXFP4 key row (64 codes, 4 scales, 12 zero)


def _e2m1_value(self, code: int) -> float:
    return float(self._lib.csa_oracle_e2m1_value(int(code) & 0xFF))


def _fp4_quantize(self, k_bits):
    """bf16 key bits [R, 128] -> MXFP4 rows [R, 80] uint8."""
    k_bits = _c(k_bits, np.uint16)
    R, ihd = k_bits.shape
    rows = np.zeros((R, FP4_ROW), dtype=np.uint8)
    _check("fp4_quantize", self._lib.csa_oracle_fp4_quantize(R, ihd, _ptr(k_bits), _ptr(rows)))
    return rows


def _fp4_dequantize(self, rows, ihd: int = 128):
    """MXFP4 rows [R, 80] -> bf16 key bits [R, 128] (exact)."""
    rows = _c(rows, np.uint8)
    R = rows.shape[0]
    k = np.zeros((R, ihd), dtype=np.uint16)
    _check("fp4_dequantize", self._lib.csa_oracle_fp4_dequantize(R, ihd, _ptr(rows), _ptr(k)))
    return k


Oracle.e2m1_value = _e2m1_value
Oracle.fp4_quantize = _fp4_quantize
Oracle.fp4_dequantize = _fp4_dequantize


def default() -> Oracle:
    """The oracle built from csa_oracle.c (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def compile_variant(src_path: str, out_path: str) -> Oracle:
    """Compile another copy of the oracle source (tests plant mistakes this way)."""
    return Oracle(build(force=True, src=src_path, out=out_path))


def num_threads(*args, **kwargs):
    return default().num_threads(*args, **kwargs)


def bf16_bits_to_f64(*args, **kwargs):
    return default().bf16_bits_to_f64(*args, **kwargs)


def n_vis(*args, **kwargs):
    return default().n_vis(*args, **kwargs)


def block_score(*args, **kwargs):
    return default().block_score(*args, **kwargs)


def indexer_scores(*args, **kwargs):
    return default().indexer_scores(*args, **kwargs)


def topk(*args, **kwargs):
    return default().topk(*args, **kwargs)


def gather(*args, **kwargs):
    return default().gather(*args, **kwargs)


def attention(*args, **kwargs):
    return default().attention(*args, **kwargs)


def _bf16_array(bits) -> np.ndarray:
    """bf16 bit patterns -> float64 (exact: a bf16 value is the top half of an f32)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def attention_partial(q, rows, scale):
    """Unnormalised attention of one part of a token's rows ([Audit 1M] D5:
    every row is the key and the value of all heads), for the sharded step's
    log-sum-exp merge.  q [H, hd] and rows [n, hd] as uint16 bf16 bits.
    Returns (O [H, hd], m [H], l [H]) in float64, natural-log units:
    m_h = max_j z_hj, l_h = sum_j exp(z_hj - m_h), O_h = sum_j exp(z_hj - m_h) row_j,
    z_hj = scale * q_h . row_j; an empty part gives (0, -inf, 0)."""
    qf = _bf16_array(q)
    rf = _bf16_array(rows).reshape(-1, qf.shape[1])
    H, hd = qf.shape
    if rf.shape[0] == 0:
        return np.zeros((H, hd)), np.full(H, -np.inf), np.zeros(H)
    z = scale * (qf @ rf.T)                      # [H, n]
    m = z.max(axis=1)
    e = np.exp(z - m[:, None])
    return e @ rf, m, e.sum(axis=1)


def combine_partials(O, m, l, sinks=None):
    """out [H, hd] = sum_p exp(m_p - M) O_p / (sum_p exp(m_p - M) l_p [+ exp(sink_h - M)]),
    M = max_p m_p, over parts p (arrays O [P, H, hd], m [P, H], l [P, H]);
    parts with m = -inf carry nothing.  Same merge as the sink identity of
    [Audit 1M] D6: the sink is one more logit with a zero value row."""
    O = np.asarray(O, dtype=np.float64)
    m = np.asarray(m, dtype=np.float64)
    l = np.asarray(l, dtype=np.float64)
    M = m.max(axis=0)                            # [H]
    if sinks is not None:
        M = np.maximum(M, np.asarray(sinks, dtype=np.float64))
    w = np.where(np.isfinite(m), np.exp(m - np.where(np.isfinite(M), M, 0.0)), 0.0)   # [P, H]
    num = (w[:, :, None] * O).sum(axis=0)
    den = (w * l).sum(axis=0)
    if sinks is not None:
        den = den + np.exp(np.asarray(sinks, dtype=np.float64) - M)
    with np.errstate(invalid="ignore", divide="ignore"):
        return np.where(den[:, None] > 0, num / den[:, None], 0.0)


def decode(*args, **kwargs):
    return default().decode(*args, **kwargs)


def hca_decode(*args, **kwargs):
    return default().hca_decode(*args, **kwargs)


def e2m1_value(*args, **kwargs):
    return default().e2m1_value(*args, **kwargs)


def fp4_quantize(*args, **kwargs):
    return default().fp4_quantize(*args, **kwargs)


def fp4_dequantize(*args, **kwargs):
    return default().fp4_dequantize(*args, **kwargs)
