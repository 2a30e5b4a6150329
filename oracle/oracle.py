"""ctypes front end of the fp64 oracle in ``ring_oracle.c``.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Arrays are numpy
float64, C-contiguous, shaped [B, H, S, d] (rows [B, H, S]).  The C code is
compiled on first use with the system ``gcc`` (OpenMP over rows / heads).

Besides the attention routines, this module holds the analytic helpers the
pages print numbers for (the "Context Parallelism" guide, section 2,
"Communication" and "Worked Example"):

* bytes rotated per ring step: K and V of one chunk, 2 * (S/P) * d_k * 2 bytes
  for BF16 -- per head; the worked example's 32K x 128 x 2 bytes x 2 = 16 MB;
* total over the P - 1 rotations, (P - 1) * 2 * (S/P) * d_k * 2 bytes
  (the example's 3 steps = 48 MB);
* KV-cache bytes per token of a multi-head model: 2 (K and V) * layers *
  heads * d_k * bytes -- 512 KB/token for the 7B / 32-head / d_k = 128 example
  at 32 layers and 2 bytes (guide section 1 and the worked example);
* score-matrix elements S^2 (guide section 1: 128K^2 = 16 billion).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

KIND_LOCAL = 0
KIND_FULL = 1
KIND_SKIP = 2

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ring_oracle.c")
_LIB = os.path.join(_HERE, "libringoracle.so")
_lock = threading.Lock()
_lib = None


def build_oracle(force: bool = False) -> str:
    """Compile ``ring_oracle.c`` into ``libringoracle.so`` (plain C, -O2, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build_oracle())
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int)
        i64p = ctypes.POINTER(ctypes.c_int64)
        c_int, c_long, c_double = ctypes.c_int, ctypes.c_long, ctypes.c_double
        lib.oracle_ring_visits.argtypes = [c_int, c_int, c_int, ip, ip]
        lib.oracle_ring_visits.restype = c_int
        lib.oracle_naive_fwd.argtypes = [dp, dp, dp, c_int, c_int, c_int, c_int,
                                         c_int, c_double, dp, dp]
        lib.oracle_naive_fwd.restype = None
        lib.oracle_naive_fwd_rows.argtypes = [dp, dp, dp, c_int, c_int, c_int,
                                              c_int, c_int, c_double, i64p,
                                              c_long, dp, dp]
        lib.oracle_naive_fwd_rows.restype = None
        lib.oracle_merge.argtypes = [dp, dp, dp, dp, c_long, c_int, dp, dp]
        lib.oracle_merge.restype = None
        lib.oracle_ring_fwd.argtypes = [dp, dp, dp, c_int, c_int, c_int, c_int,
                                        c_int, c_int, c_double, dp, dp, ip]
        lib.oracle_ring_fwd.restype = c_int
        lib.oracle_bwd.argtypes = [dp, dp, dp, dp, c_int, c_int, c_int, c_int,
                                   c_int, c_double, dp, dp, dp, dp, dp]
        lib.oracle_bwd.restype = None
        lib.oracle_bwd_dq_rows.argtypes = [dp, dp, dp, dp, c_int, c_int, c_int,
                                           c_int, c_int, c_double, i64p, c_long,
                                           dp, dp]
        lib.oracle_bwd_dq_rows.restype = None
        lib.oracle_partial.argtypes = [dp, c_long, c_long, dp, dp, c_long, c_long,
                                       c_int, c_int, c_double, dp, dp]
        lib.oracle_partial.restype = None
        _lib = lib
        return lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a: np.ndarray, ty=ctypes.c_double):
    return a.ctypes.data_as(ctypes.POINTER(ty))


def _shape4(q):
    if q.ndim != 4:
        raise ValueError("expected [B, H, S, d]")
    return q.shape


def ring_visits(P: int, causal: bool, i: int):
    """Visit list of query chunk i: list of (t, j, kind) for t = 0..P-1."""
    lib = _load()
    js = (ctypes.c_int * P)()
    ks = (ctypes.c_int * P)()
    n = lib.oracle_ring_visits(P, int(bool(causal)), i, js, ks)
    if n < 0:
        raise ValueError("bad ring arguments")
    return [(t, js[t], ks[t]) for t in range(P)]


def naive_fwd(q, k, v, causal: bool, scale: float):
    """Definition over whole rows -> (O [B,H,S,d], LSE [B,H,S]) in fp64."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, S, d = _shape4(q)
    o = np.empty_like(q)
    lse = np.empty((B, H, S), dtype=np.float64)
    _load().oracle_naive_fwd(_ptr(q), _ptr(k), _ptr(v), B, H, S, d,
                             int(bool(causal)), float(scale), _ptr(o), _ptr(lse))
    return o, lse


def naive_fwd_rows(q, k, v, causal: bool, scale: float, rows):
    """Definition for selected flat rows (index bh * S + r) -> (O [n,d], LSE [n])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, S, d = _shape4(q)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    if rows.size and (rows.min() < 0 or rows.max() >= B * H * S):
        raise ValueError("row index out of range")
    o = np.empty((rows.size, d), dtype=np.float64)
    lse = np.empty(rows.size, dtype=np.float64)
    _load().oracle_naive_fwd_rows(_ptr(q), _ptr(k), _ptr(v), B, H, S, d,
                                  int(bool(causal)), float(scale),
                                  _ptr(rows, ctypes.c_int64), rows.size,
                                  _ptr(o), _ptr(lse))
    return o, lse


def merge(o_a, lse_a, o_b, lse_b):
    """Log-sum-exp merge of two partials, row-wise -> (O, LSE)."""
    o_a, o_b = _f64(o_a), _f64(o_b)
    lse_a, lse_b = _f64(lse_a), _f64(lse_b)
    if o_a.shape != o_b.shape or lse_a.shape != lse_b.shape:
        raise ValueError("shape mismatch")
    d = o_a.shape[-1]
    rows = lse_a.size
    if o_a.size != rows * d:
        raise ValueError("O and LSE disagree")
    o = np.empty_like(o_a)
    lse = np.empty_like(lse_a)
    _load().oracle_merge(_ptr(o_a), _ptr(lse_a), _ptr(o_b), _ptr(lse_b), rows, d,
                         _ptr(o), _ptr(lse))
    return o, lse


def ring_fwd(q, k, v, P: int, causal: bool, scale: float):
    """Ring schedule taken literally -> (O, LSE, visit_log [P, P, 3])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, S, d = _shape4(q)
    o = np.empty_like(q)
    lse = np.empty((B, H, S), dtype=np.float64)
    log = np.zeros((P, P, 3), dtype=np.int32)
    rc = _load().oracle_ring_fwd(_ptr(q), _ptr(k), _ptr(v), B, H, S, d, P,
                                 int(bool(causal)), float(scale), _ptr(o), _ptr(lse),
                                 _ptr(log, ctypes.c_int))
    if rc != 0:
        raise ValueError("bad ring arguments (S must divide into P equal chunks)")
    return o, lse, log


def partial(q_rows, r0: int, k_rows, v_rows, c0: int, causal: bool, scale: float):
    """One ring step's partial: query rows at global positions r0.. against
    keys at c0.. (one head, [n, d] each) -> (O [nq, d], LSE [nq])."""
    q_rows, k_rows, v_rows = _f64(q_rows), _f64(k_rows), _f64(v_rows)
    nq, d = q_rows.shape
    nk = k_rows.shape[0]
    if k_rows.shape != (nk, d) or v_rows.shape != (nk, d):
        raise ValueError("shape mismatch")
    o = np.empty((nq, d), dtype=np.float64)
    lse = np.empty(nq, dtype=np.float64)
    _load().oracle_partial(_ptr(q_rows), r0, nq, _ptr(k_rows), _ptr(v_rows), c0, nk, d,
                           int(bool(causal)), float(scale), _ptr(o), _ptr(lse))
    return o, lse


def bwd(q, k, v, dO, causal: bool, scale: float):
    """Plain derivative of L = sum(dO * O) -> (dQ, dK, dV, LSE, D)."""
    q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
    B, H, S, d = _shape4(q)
    dq = np.empty_like(q)
    dk = np.empty_like(q)
    dv = np.empty_like(q)
    lse = np.empty((B, H, S), dtype=np.float64)
    D = np.empty((B, H, S), dtype=np.float64)
    _load().oracle_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(dO), B, H, S, d,
                       int(bool(causal)), float(scale), _ptr(dq), _ptr(dk), _ptr(dv),
                       _ptr(lse), _ptr(D))
    return dq, dk, dv, lse, D


def bwd_dq_rows(q, k, v, dO, causal: bool, scale: float, rows):
    """dQ and D for selected flat query rows -> (dQ [n,d], D [n])."""
    q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
    B, H, S, d = _shape4(q)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    if rows.size and (rows.min() < 0 or rows.max() >= B * H * S):
        raise ValueError("row index out of range")
    dq = np.empty((rows.size, d), dtype=np.float64)
    D = np.empty(rows.size, dtype=np.float64)
    _load().oracle_bwd_dq_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(dO), B, H, S, d,
                               int(bool(causal)), float(scale),
                               _ptr(rows, ctypes.c_int64), rows.size, _ptr(dq), _ptr(D))
    return dq, D


# ---------------------------------------------------------------------------
# Grouped-query attention: H query heads share H_kv key/value heads; query
# head h reads key/value head h // (H / H_kv).  The pages name GQA as the
# case where ring attention, unlike head-partitioned schemes, does not depend
# on the head count ("Training Long-Context Models Without OOM: Ring
# Attention", section "Ring Attention vs. DeepSpeed Ulysses (All-to-All)").
# The definition is multi-head attention on K and V with each head repeated
# for its group; the gradient of a shared K or V head is the sum over its
# group.
# ---------------------------------------------------------------------------

def _repeat_kv(x, H: int):
    x = _f64(x)
    Hkv = x.shape[1]
    if H % Hkv:
        raise ValueError("H must be a multiple of H_kv")
    return np.ascontiguousarray(np.repeat(x, H // Hkv, axis=1))


def naive_fwd_gqa(q, k, v, causal: bool, scale: float):
    """GQA forward -> (O [B,H,S,d], LSE [B,H,S]); k, v are [B,H_kv,S,d]."""
    H = np.asarray(q).shape[1]
    return naive_fwd(q, _repeat_kv(k, H), _repeat_kv(v, H), causal, scale)


def naive_fwd_rows_gqa(q, k, v, causal: bool, scale: float, rows):
    H = np.asarray(q).shape[1]
    return naive_fwd_rows(q, _repeat_kv(k, H), _repeat_kv(v, H), causal, scale, rows)


def bwd_gqa(q, k, v, dO, causal: bool, scale: float):
    """GQA backward -> (dQ [B,H,S,d], dK, dV [B,H_kv,S,d])."""
    q = _f64(q)
    B, H, S, d = q.shape
    Hkv = np.asarray(k).shape[1]
    dq, dk, dv, _, _ = bwd(q, _repeat_kv(k, H), _repeat_kv(v, H), dO, causal, scale)
    G = H // Hkv
    return dq, dk.reshape(B, Hkv, G, S, d).sum(axis=2), dv.reshape(B, Hkv, G, S, d).sum(axis=2)


# ---------------------------------------------------------------------------
# Analytic helpers ("Context Parallelism" guide, section 2)
# ---------------------------------------------------------------------------

def ring_step_bytes(S: int, P: int, d_k: int, elem_bytes: int = 2, heads: int = 1) -> int:
    """K and V of one chunk: 2 * (S/P) * d_k * elem_bytes per head."""
    if S % P:
        raise ValueError("S must divide into P chunks")
    return 2 * (S // P) * d_k * elem_bytes * heads


def ring_total_bytes(S: int, P: int, d_k: int, elem_bytes: int = 2, heads: int = 1) -> int:
    """All P - 1 rotations: (P - 1) * 2 * (S/P) * d_k * elem_bytes per head."""
    return (P - 1) * ring_step_bytes(S, P, d_k, elem_bytes, heads)


def kv_cache_bytes_per_token(layers: int, heads: int, d_k: int, elem_bytes: int = 2) -> int:
    """K and V of every layer and head for one token."""
    return 2 * layers * heads * d_k * elem_bytes


def score_matrix_elements(S: int) -> int:
    """Entries of one head's S x S score matrix."""
    return S * S


def attention_flops(B: int, H: int, S: int, d: int, causal: bool) -> int:
    """Forward FLOPs counted as 4 d per allowed (query, key) pair (QK^T and
    PV, one multiply-add = 2 FLOPs each).  Causal counts pairs c <= r."""
    pairs = S * (S + 1) // 2 if causal else S * S
    return 4 * d * pairs * B * H


# ---------------------------------------------------------------------------
# Whole-head passes with a matrix product as the step (PyTorch, fp64, CPU)
# ---------------------------------------------------------------------------
# The C routines above take one dot product at a time: minutes per head at
# S = 32768, hours at 131072.  The two routines below take the same
# definition with query rows batched into blocks, so that each row's score
# vector comes out of one fp64 matrix product (a library primitive); every
# other step is the definition written out on those vectors, row by row:
#     s_rc  = scale <q_r, k_c> on the allowed set (c <= r when causal)
#     M_r   = max_c s_rc,   L_r = sum_c exp(s_rc - M_r),   LSE_r = M_r + ln L_r
#     P_rc  = exp(s_rc - M_r) / L_r  (= exp(s_rc - LSE_r)),   O_r = sum_c P_rc v_c
#     dP_rc = <dO_r, v_c>,   D_r = sum_c P_rc dP_rc,   dS_rc = P_rc (dP_rc - D_r)
#     dK_c  = scale sum_r dS_rc q_r,   dV_c = sum_r P_rc dO_r.
# The parity tests use them where LSE_r and D_r of every row of a long head
# are needed (sampled key rows of dK and dV need every query row r >= c).

def _heads64(x):
    import torch
    t = torch.as_tensor(np.asarray(x, dtype=np.float64))
    if t.ndim != 4:
        raise ValueError("expected [B, H, S, d]")
    return t


def _row_block_scores(Qb, K, r0, causal, scale):
    """Scores of query rows r0 .. r0 + len(Qb) - 1 against keys 0 .. len(K) - 1,
    with the keys c > r set to -inf when causal."""
    import torch
    s = (Qb @ K.T) * scale
    if causal:
        r = torch.arange(r0, r0 + Qb.shape[0]).unsqueeze(1)
        c = torch.arange(K.shape[0]).unsqueeze(0)
        s.masked_fill_(c > r, float("-inf"))
    return s


def naive_fwd_blocked(q, k, v, causal: bool, scale: float, block: int = 256):
    """The definition over whole [B, H, S, d] tensors, query rows in blocks
    -> (O, LSE) as numpy float64."""
    import torch
    Q, K, V = _heads64(q), _heads64(k), _heads64(v)
    B, H, S, d = Q.shape
    O = torch.empty_like(Q)
    LSE = torch.empty((B, H, S), dtype=torch.float64)
    for b in range(B):
        for h in range(H):
            for r0 in range(0, S, block):
                r1 = min(S, r0 + block)
                kmax = r1 if causal else S          # keys past the block's last row are masked
                s = _row_block_scores(Q[b, h, r0:r1], K[b, h, :kmax], r0, causal, scale)
                M = s.max(dim=1, keepdim=True).values
                e = torch.exp(s - M)
                L = e.sum(dim=1, keepdim=True)
                O[b, h, r0:r1] = (e / L) @ V[b, h, :kmax]
                LSE[b, h, r0:r1] = (M + torch.log(L)).squeeze(1)
    return O.numpy(), LSE.numpy()


def bwd_dkdv_rows(q, k, v, dO, causal: bool, scale: float, keys, block: int = 256):
    """dK and dV at chosen key positions of ONE head ([1, 1, S, d] inputs),
    with LSE_r and D_r of every query row computed here from the definition.
    Returns (dK [n, d], dV [n, d], LSE [S], D [S]) as numpy float64."""
    import torch
    Q, K, V, dOt = (_heads64(x) for x in (q, k, v, dO))
    if Q.shape[:2] != (1, 1):
        raise ValueError("one head at a time: inputs shaped [1, 1, S, d]")
    Q, K, V, dOt = Q[0, 0], K[0, 0], V[0, 0], dOt[0, 0]
    S, d = Q.shape
    keys = torch.as_tensor(np.asarray(keys, dtype=np.int64))
    if keys.numel() and (int(keys.min()) < 0 or int(keys.max()) >= S):
        raise ValueError("key index out of range")
    dK = torch.zeros((keys.numel(), d), dtype=torch.float64)
    dV = torch.zeros((keys.numel(), d), dtype=torch.float64)
    LSE = torch.empty(S, dtype=torch.float64)
    Dv = torch.empty(S, dtype=torch.float64)
    for r0 in range(0, S, block):
        r1 = min(S, r0 + block)
        kmax = r1 if causal else S
        s = _row_block_scores(Q[r0:r1], K[:kmax], r0, causal, scale)
        M = s.max(dim=1, keepdim=True).values
        e = torch.exp(s - M)
        L = e.sum(dim=1, keepdim=True)
        Pm = e / L
        dP = dOt[r0:r1] @ V[:kmax].T
        D = (Pm * dP).sum(dim=1, keepdim=True)
        LSE[r0:r1] = (M + torch.log(L)).squeeze(1)
        Dv[r0:r1] = D.squeeze(1)
        sel = torch.nonzero(keys < kmax).squeeze(1)     # keys these rows can see
        if sel.numel() == 0:
            continue
        cols = keys[sel]
        Psel = Pm[:, cols]
        dS = Psel * (dP[:, cols] - D)
        dK[sel] += scale * (dS.T @ Q[r0:r1])
        dV[sel] += Psel.T @ dOt[r0:r1]
    return dK.numpy(), dV.numpy(), LSE.numpy(), Dv.numpy()


# ---------------------------------------------------------------------------
# Rounding model of a bf16-storage backward (PyTorch, fp64, CPU)
# ---------------------------------------------------------------------------
# The plain derivative above is exact; a backward whose tensors are stored in
# bf16 cannot reach it.  This routine evaluates the same derivative in fp64
# with an exact bf16 rounding (round to nearest even) applied at the four
# places where the stored format is bf16:
#   O      -- the forward's output, which D_r = <dO_r, O_r> is formed from
#             (activations kept for the backward pass, "Training
#             Long-Context Models Without OOM: Ring Attention", section
#             "Diagnosing the Sequence-Length OOM");
#   P      -- the probabilities entering dV = P^T dO;
#   dS     -- entering dQ = scale dS K and dK = scale dS^T Q;
#   dQ, dK, dV -- the outputs.
# Its distance from the exact derivative is the error that storage alone
# causes; the parity tests of stress inputs allow that much on top of the
# gradient tolerance.  With round_bf16=False every rounding is the identity
# and the routine is the plain derivative again.

def _bf16_rne(t):
    """fp64 -> nearest bf16 value (ties to even), returned as fp64.  Done on
    the bit pattern of the fp32 value nearest t; fp64 inputs here are bf16
    values times O(1) factors, so the fp32 step never decides a tie."""
    import torch
    f = t.to(torch.float32).contiguous()
    bits = f.view(torch.int32).to(torch.int64) & 0xFFFFFFFF
    lsb = (bits >> 16) & 1
    rounded = ((bits + 0x7FFF + lsb) >> 16) << 16
    out = (rounded & 0xFFFFFFFF).to(torch.int64)
    out = torch.where(out >= 2 ** 31, out - 2 ** 32, out).to(torch.int32)
    return out.view(torch.float32).to(torch.float64)


def bwd_bf16_rounding_model(q, k, v, dO, causal: bool, scale: float, round_bf16: bool = True):
    """(dQ, dK, dV) of whole [B, H, S, d] tensors with bf16 storage of O, P,
    dS and the outputs (see above) -> numpy float64.  Small shapes only
    (S x S matrices per head)."""
    import torch
    Q, K, V, dOt = (_heads64(x) for x in (q, k, v, dO))
    B, H, S, d = Q.shape
    rnd = _bf16_rne if round_bf16 else (lambda t: t)
    dQ, dK, dV = torch.empty_like(Q), torch.empty_like(Q), torch.empty_like(Q)
    mask = torch.triu(torch.ones(S, S, dtype=torch.bool), diagonal=1) if causal else None
    for b in range(B):
        for h in range(H):
            s = (Q[b, h] @ K[b, h].T) * scale
            if causal:
                s.masked_fill_(mask, float("-inf"))
            M = s.max(dim=1, keepdim=True).values
            e = torch.exp(s - M)
            Pm = e / e.sum(dim=1, keepdim=True)
            O = rnd(Pm @ V[b, h])
            D = (dOt[b, h] * O).sum(dim=1, keepdim=True)
            dS = Pm * (dOt[b, h] @ V[b, h].T - D)
            dV[b, h] = rnd(rnd(Pm).T @ dOt[b, h])
            dQ[b, h] = rnd(scale * (rnd(dS) @ K[b, h]))
            dK[b, h] = rnd(scale * (rnd(dS).T @ Q[b, h]))
    return dQ.numpy(), dK.numpy(), dV.numpy()
