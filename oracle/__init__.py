"""CPU oracle for the DSpark vocabulary-wide hot path (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s ``cpu_baseline``
and reference legs may import this package.  It wraps ``dspark_oracle.c`` (plain
single-threaded C, fp64) with ctypes; it never imports the CUDA package and the
CUDA package never imports it.

Arrays are numpy arrays.  bf16 data is passed as ``uint16`` bit patterns, fp32 as
``float32``; the C side converts both exactly to double.

Parity pins live in ``tests/test_oracle_*.py``; see the C file header for the
list and for the sources (P1..P4 are the four DSpark pages, cited by title and
section).
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

F32, BF16 = 0, 1
TILE, CHUNK = 1024, 32  # the library's vocabulary tile and chunk sizes
P_SAMPLE_CHUNK, P_SAMPLE_INCHUNK, P_ACCEPT = 1, 2, 3
P_RESID_CHUNK, P_RESID_INCHUNK, P_BONUS_CHUNK, P_BONUS_INCHUNK, P_ELEM_GUMBEL = 4, 5, 6, 7, 8

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dspark_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = C.CDLL(_LIB)
        vp, i32, i64, u32, u64, dbl = C.c_void_p, C.c_int, C.c_int64, C.c_uint32, C.c_uint64, C.c_double
        L.oracle_philox4x32_10.argtypes = [vp, vp, vp]
        L.oracle_philox_word.argtypes = [u64, u32, u32, u32, u32]
        L.oracle_philox_word.restype = u32
        L.oracle_uniform.argtypes = [u64, u32, u32, u32, u32]
        L.oracle_uniform.restype = dbl
        L.oracle_markov_logits.argtypes = [i32, i32, i32, i32, vp, vp, vp, i32, dbl, vp]
        L.oracle_argmax.argtypes = [vp, i32, vp]
        L.oracle_argmax.restype = i32
        L.oracle_chunk_gumbel.argtypes = [vp, i32, i32, u64, i32, i32, i32, i32, vp, vp]
        L.oracle_chunk_gumbel.restype = i32
        L.oracle_gumbel_elem.argtypes = [vp, i32, u64, i32, i32, vp]
        L.oracle_gumbel_elem.restype = i32
        L.oracle_sample_request.argtypes = [i32, i32, i32, i32, i32, dbl, u64, i32, i32, vp, vp, vp, i32, i32,
                                            vp, vp, vp, vp, dbl]
        L.oracle_verify_request.argtypes = [i32, i32, i32, i32, i32, i32, dbl, u64, i32, i32, i32, vp, vp, vp,
                                            i32, i32, vp, vp, vp, vp, i32, vp, vp, vp, dbl, vp]
        L.oracle_sample_request_head.argtypes = [i32, i32, i32, i32, i32, dbl, u64, i32, i32, vp, vp, vp, i32, i32,
                                                 i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, dbl]
        L.oracle_verify_request.restype = i32
        L.oracle_tv_row.argtypes = [i32, i32, vp, vp, vp]
        L.oracle_tv_row.restype = dbl
        L.oracle_eval_mask_tau.argtypes = [i32, i32, vp, vp, vp]
        L.oracle_eval_mask_tau.restype = dbl
        L.oracle_schedule.argtypes = [i32, i32, vp, i32, vp, vp, vp, vp]
        L.oracle_schedule.restype = i32
        L.oracle_theta_schedule.argtypes = [i32, vp, vp, vp, vp]
        L.oracle_theta_schedule.restype = i32
        L.oracle_trials_sampler.argtypes = [i32, i32, vp, u64, i64, i32, vp]
        L.oracle_trials_spec_one.argtypes = [i32, i32, i32, dbl, vp, vp, u64, i64, vp, vp]
        L.oracle_trials_spec_block.argtypes = [i32, i32, i32, i32, i32, dbl, vp, vp, vp, i32, vp, u64, i64, vp]
        _lib = L
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(C.c_void_p)


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    raise TypeError(f"oracle takes float32 or bf16-as-uint16, got {a.dtype}")


def to_f64(a: np.ndarray) -> np.ndarray:
    """Exact conversion of a float32 or bf16-bits array to float64 (format change only)."""
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


# ----------------------------------------------------------------- randomness
def philox4x32_10(ctr, key) -> tuple:
    c = np.asarray(ctr, dtype=np.uint32).copy()
    k = np.asarray(key, dtype=np.uint32).copy()
    out = np.zeros(4, dtype=np.uint32)
    lib().oracle_philox4x32_10(_p(c), _p(k), _p(out))
    return tuple(int(x) for x in out)


def philox_word(seed: int, j: int, i: int, purpose: int, n: int) -> int:
    return int(lib().oracle_philox_word(seed, j, i, purpose, n))


def uniform(seed: int, j: int, i: int, purpose: int, n: int) -> float:
    return float(lib().oracle_uniform(seed, j, i, purpose, n))


# ----------------------------------------------------------------- sampler
def markov_logits(base_row: np.ndarray, W1: np.ndarray | None, W2: np.ndarray | None, prev: int,
                  softcap: float = 0.0) -> np.ndarray:
    """z = cap(base) + W2 W1[prev] in fp64; cap(b) = s tanh(b / s) with s = softcap > 0, else b."""
    V = base_row.shape[-1]
    r = 0 if W1 is None else W1.shape[1]
    z = np.zeros(V, dtype=np.float64)
    w_dt = _dtype_code(W1) if r else F32
    w1 = _p(W1) if r else None
    w2 = _p(W2) if r else None
    lib().oracle_markov_logits(V, r, _dtype_code(base_row), w_dt, _p(base_row), w1, w2, int(prev), float(softcap),
                               _p(z))
    return z


def block_logits(base: np.ndarray, W1, W2, anchor, tokens, softcap: float = 0.0) -> np.ndarray:
    """Teacher-forced z[j, i] = markov_logits(base[j, i], W1, W2, prev_{j,i}) with prev_{j,0} = anchor[j] and
    prev_{j,i} = tokens[j, i - 1] (P1 section on build_markov_head, apply_block_logits), in fp64."""
    B, gamma, V = base.shape
    z = np.empty((B, gamma, V))
    for j in range(B):
        for i in range(gamma):
            prev = int(anchor[j]) if i == 0 else int(tokens[j, i - 1])
            z[j, i] = markov_logits(base[j, i], W1, W2, prev, softcap)
    return z


def argmax(z: np.ndarray):
    z = np.ascontiguousarray(z, dtype=np.float64)
    m = np.zeros(1)
    x = lib().oracle_argmax(_p(z), z.shape[0], _p(m))
    return int(x), float(m[0])


def chunk_gumbel(lw: np.ndarray, seed: int, j: int, i: int, CS: int = CHUNK, p_chunk=P_SAMPLE_CHUNK,
                 p_inchunk=P_SAMPLE_INCHUNK):
    """The chunk-Gumbel draw (the draft sampler's purposes by default; verify's corrections use the
    RESID / BONUS purposes).  Returns (x, margin, lse)."""
    lw = np.ascontiguousarray(lw, dtype=np.float64)
    m, lse = np.zeros(1), np.zeros(1)
    x = lib().oracle_chunk_gumbel(_p(lw), lw.shape[0], CS, seed, j, i, p_chunk, p_inchunk, _p(m), _p(lse))
    return int(x), float(m[0]), float(lse[0])


def gumbel_elem(lw: np.ndarray, seed: int, j: int, i: int):
    lw = np.ascontiguousarray(lw, dtype=np.float64)
    m = np.zeros(1)
    x = lib().oracle_gumbel_elem(_p(lw), lw.shape[0], seed, j, i, _p(m))
    return int(x), float(m[0])


def sample_request(base: np.ndarray, W1, W2, anchor: int, j: int, T: float, seed: int, TS: int, row=None,
                   CS: int = CHUNK, softcap: float = 0.0):
    """One request of dspark_markov_sample_block.  base: [B, gamma, V]; j is the
    request index (random stream); `row` selects the data block (default j)."""
    B, gamma, V = base.shape
    r = 0 if W1 is None else W1.shape[1]
    blk = np.ascontiguousarray(base[j if row is None else row])
    tok = np.zeros(gamma, dtype=np.int32)
    lse, zx, mg = np.zeros(gamma), np.zeros(gamma), np.zeros(gamma)
    w_dt = _dtype_code(W1) if r else F32
    lib().oracle_sample_request(V, r, gamma, TS, CS, float(T), seed, _dtype_code(base), w_dt, _p(blk),
                                _p(W1) if r else None, _p(W2) if r else None, int(anchor), int(j),
                                _p(tok), _p(lse), _p(zx), _p(mg), float(softcap))
    return tok, lse, zx, mg


HEAD_VANILLA, HEAD_GATED, HEAD_RNN = 0, 1, 2


def sample_request_head(base: np.ndarray, W1, W2, anchor: int, j: int, T: float, seed: int, TS: int, kind: int,
                        hidden: np.ndarray, Wg, Wc=None, Wo=None, CS: int = CHUNK, softcap: float = 0.0):
    """One request of the Gated / RNN head sampler (P1 section 3.7).  hidden [B, gamma, d] (the request's
    rows are used) and the head weights share W1's dtype.  Returns (tokens, lse, z_at_tok, margins,
    head vectors [gamma, r])."""
    B, gamma, V = base.shape
    r = W1.shape[1]
    d = hidden.shape[-1]
    blk = np.ascontiguousarray(base[j])
    hrow = np.ascontiguousarray(hidden[j])
    tok = np.zeros(gamma, dtype=np.int32)
    lse, zx, mg = np.zeros(gamma), np.zeros(gamma), np.zeros(gamma)
    u = np.zeros((gamma, r))
    w_dt = _dtype_code(W1)
    lib().oracle_sample_request_head(V, r, gamma, TS, CS, float(T), seed, _dtype_code(base), w_dt, _p(blk), _p(W1),
                                     _p(W2), int(anchor), int(j), int(kind), int(d), _p(hrow), _p(Wg),
                                     _p(Wc) if Wc is not None else None, _p(Wo) if Wo is not None else None,
                                     _p(tok), _p(lse), _p(zx), _p(mg), _p(u), float(softcap))
    return tok, lse, zx, mg, u


def sample_block(base, W1, W2, anchor, T, seed, TS, requests=None, CS: int = CHUNK):
    """Oracle of dspark_markov_sample_block for the listed requests (default all)."""
    B, gamma, V = base.shape
    req = range(B) if requests is None else requests
    out = {}
    for j in req:
        out[int(j)] = sample_request(base, W1, W2, int(anchor[j]), int(j), T, seed, TS, CS=CS)
    return out


# ----------------------------------------------------------------- verify
def verify_request(base, W1, W2, anchor: int, j: int, tokens, draft_lse, z_at_tok, target, L: int,
                   T: float, seed: int, TS: int, row=None, CS: int = CHUNK, softcap: float = 0.0, head_vec=None):
    """One request of dspark_verify.  base [B,gamma,V], target [B,gamma_t,V];
    tokens/draft_lse/z_at_tok: this request's gamma entries (int32 / float32);
    j is the request index (random stream); `row` selects the data (default j)."""
    B, gamma, V = base.shape
    gamma_t = target.shape[1]
    r = 0 if W1 is None else W1.shape[1]
    rw = j if row is None else row
    bblk = np.ascontiguousarray(base[rw])
    tblk = np.ascontiguousarray(target[rw])
    tok = np.ascontiguousarray(tokens, dtype=np.int32)
    dl = np.ascontiguousarray(draft_lse, dtype=np.float32)
    zx = np.ascontiguousarray(z_at_tok, dtype=np.float32)
    corr = np.zeros(1, dtype=np.int32)
    mm = np.zeros(1)
    fb = np.zeros(1, dtype=np.int32)
    hv = None if head_vec is None else np.ascontiguousarray(head_vec, dtype=np.float64)
    w_dt = _dtype_code(W1) if r else F32
    n = lib().oracle_verify_request(V, r, gamma, gamma_t, TS, CS, float(T), seed, _dtype_code(base), w_dt,
                                    _dtype_code(target), _p(bblk), _p(W1) if r else None,
                                    _p(W2) if r else None, int(anchor), int(j), _p(tok), _p(dl), _p(zx),
                                    _p(tblk), int(L), _p(corr), _p(mm), _p(fb), float(softcap),
                                    _p(hv) if hv is not None else None)
    return int(n), int(corr[0]), float(mm[0]), int(fb[0])


# ----------------------------------------------------------------- TV / eval mask
def tv_row(d_row: np.ndarray, t_row: np.ndarray):
    d_row = np.ascontiguousarray(d_row)
    t_row = np.ascontiguousarray(t_row)
    assert d_row.dtype == t_row.dtype
    chk = np.zeros(1)
    acc = lib().oracle_tv_row(d_row.shape[0], _dtype_code(d_row), _p(d_row), _p(t_row), _p(chk))
    return float(acc), float(chk[0])


def eval_mask_tau(acc: np.ndarray, keep: int, pos_valid: np.ndarray | None):
    acc = np.ascontiguousarray(acc, dtype=np.float64)
    mask = np.zeros_like(acc)
    pv = None if pos_valid is None else np.ascontiguousarray(pos_valid, dtype=np.uint8)
    tau = lib().oracle_eval_mask_tau(acc.shape[0], int(keep), _p(pv) if pv is not None else None, _p(acc), _p(mask))
    return mask, float(tau)


# ----------------------------------------------------------------- schedulers
def tv_l1_loss(acc: np.ndarray, mask: np.ndarray, decay: float = 4.0):
    """L1 term on accept rates (P1 section 3.9): l1 = 2 (1 - acc) per position, weights
    w_k = exp(-(k-1)/decay) for positions k = 1..gamma (the last axis); returns (l1, sum w mask l1,
    sum w mask) in fp64."""
    acc = np.asarray(acc, dtype=np.float64)
    mask = np.asarray(mask, dtype=np.float64)
    l1 = 2.0 * (1.0 - acc)
    w = np.exp(-np.arange(acc.shape[-1]) / decay)
    return l1, float(np.sum(w * mask * l1)), float(np.sum(w * mask))


def schedule(conf: np.ndarray, budget: int):
    conf = np.ascontiguousarray(conf, dtype=np.float32)
    B, gamma = conf.shape
    L = np.zeros(B, dtype=np.int32)
    off = np.zeros(B + 1, dtype=np.int32)
    obj, mg = np.zeros(1), np.zeros(1)
    rc = lib().oracle_schedule(B, gamma, _p(conf), int(budget), _p(L), _p(off), _p(obj), _p(mg))
    if rc != 0:
        raise ValueError("budget < B")
    return L, off, float(obj[0]), float(mg[0])


def theta_schedule(c, sps, with_margin: bool = False):
    """Throughput-aware prefix choice in fp64 (P4 section 5.1): returns (ell, Theta_0..Theta_gamma
    as far as the causal search evaluated them, NaN after) and, with_margin, the smallest relative
    gap between two Theta values the search compared."""
    c = np.ascontiguousarray(c, dtype=np.float64)
    sps = np.ascontiguousarray(sps, dtype=np.float64)
    gamma = c.shape[0]
    assert sps.shape[0] >= gamma + 1
    th = np.zeros(gamma + 1)
    mg = np.zeros(1)
    ell = lib().oracle_theta_schedule(gamma, _p(c), _p(sps), _p(th), _p(mg))
    if with_margin:
        return int(ell), th, float(mg[0])
    return int(ell), th


# ----------------------------------------------------------------- trial drivers
def trials_sampler(lw, seed, ntrials, variant=0, CS: int = CHUNK):
    """Draw counts over ntrials (trial n = request n): variant 0 = chunk-Gumbel with the correction
    purposes, 1 = per-element Gumbel-max, 2 = chunk-Gumbel with the sampling purposes."""
    lw = np.ascontiguousarray(lw, dtype=np.float64)
    counts = np.zeros(lw.shape[0], dtype=np.int64)
    lib().oracle_trials_sampler(lw.shape[0], CS, _p(lw), seed, int(ntrials), int(variant), _p(counts))
    return counts


def trials_spec_one(zd, zt, T, TS, seed, ntrials, CS: int = CHUNK):
    zd = np.ascontiguousarray(zd, dtype=np.float32)
    zt = np.ascontiguousarray(zt, dtype=np.float32)
    em = np.zeros(zd.shape[0], dtype=np.int64)
    na = np.zeros(1, dtype=np.int64)
    lib().oracle_trials_spec_one(zd.shape[0], TS, CS, float(T), _p(zd), _p(zt), seed, int(ntrials), _p(em), _p(na))
    return em, int(na[0])


def trials_spec_block(base_req, W1, W2, anchor, target_req, T, TS, seed, ntrials, CS: int = CHUNK):
    """fp32 blocks: base_req/target_req [gamma, V], W1/W2 [V, r].  Returns the
    histogram of the accepted length over ntrials independent draws."""
    base_req = np.ascontiguousarray(base_req, dtype=np.float32)
    target_req = np.ascontiguousarray(target_req, dtype=np.float32)
    W1 = np.ascontiguousarray(W1, dtype=np.float32)
    W2 = np.ascontiguousarray(W2, dtype=np.float32)
    gamma, V = base_req.shape
    hist = np.zeros(gamma + 1, dtype=np.int64)
    lib().oracle_trials_spec_block(V, W1.shape[1], gamma, TS, CS, float(T), _p(base_req), _p(W1), _p(W2), int(anchor),
                                   _p(target_req), seed, int(ntrials), _p(hist))
    return hist
