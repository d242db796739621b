"""CPU oracle for speculative-decoding verification and DSpark drafting -- TEST INFRASTRUCTURE.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
this package.  It wraps ``oracle.c`` (plain double-precision C, see ``oracle.h`` for the sources each
function follows) through ctypes and shares nothing with the CUDA library.

All array arguments are numpy arrays on the host; logits are float32 (bf16 inputs widened exactly).
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_SOURCES = [os.path.join(_HERE, "oracle.c")]
_HEADER = os.path.join(_HERE, "oracle.h")
_lock = threading.Lock()
_lib = None

TAG_DRAFT, TAG_ACCEPT, TAG_RESID, TAG_BONUS = 0, 1, 2, 3
TAG_FINE = 4  # added to a race tag: the stream of the low bits of its uniforms
OK, ERR_ARGS, ERR_TOKEN, ERR_NAN, ERR_ZERO_Q = 0, 1, 2, 3, 4
RACE_RESIDUAL, RACE_BONUS, RACE_RESIDUAL_EMPTY = 0, 1, 2


class VerifyResult(C.Structure):
    _fields_ = [
        ("accepted_len", C.c_int32),
        ("correction", C.c_int32),
        ("race_kind", C.c_int32),
        ("status", C.c_int32),
        ("decision_margin", C.c_double),
        ("race_margin", C.c_double),
    ]


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` with the host C compiler (portable flags, no -march)."""
    newest = max(os.path.getmtime(p) for p in _SOURCES + [_HEADER])
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= newest:
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math", "-ffp-contract=off",
           "-o", tmp] + _SOURCES + ["-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = C.CDLL(build())
        P = C.c_void_p
        i32, i64, u32, u64, f64 = C.c_int32, C.c_int64, C.c_uint32, C.c_uint64, C.c_double
        sig = {
            "orc_philox4x32_10": (None, [P, P, P]),
            "orc_random_word": (u32, [u64, u64, u32, u32, u64]),
            "orc_uniform": (f64, [u64, u64, u32, u32, u64]),
            "orc_race_uniform": (f64, [u64, u64, u32, u32, u64]),
            "orc_row_stats": (C.c_int, [P, i64, P, P]),
            "orc_overlap": (f64, [P, P, i64]),
            "orc_expected_words": (f64, [f64, C.c_int]),
            "orc_speedup": (f64, [f64, C.c_int, f64]),
            "orc_sample_race": (C.c_int, [P, i64, u64, u64, u32, u32, P, P]),
            "orc_sample_draft_batch": (C.c_int, [P, i64, i64, P, P, i32, u64, P, P]),
            "orc_lmhead_logits": (C.c_int, [P, P, i64, i64, i64, P]),
            "orc_race_shard": (C.c_int, [P, P, i64, i64, C.c_int, f64, f64, f64, f64, f64,
                                         u64, u64, u32, u32, P, P]),
            "orc_verify_token_request": (C.c_int, [P, P, i64, i64, P, i32, u64, u64, P, P]),
            "orc_verify_block_request": (C.c_int, [P, P, i64, i64, P, i32, u64, u64, P, P, P]),
            "orc_verify_batch": (C.c_int, [C.c_int, P, P, i64, i64, P, P, P, P, i32, u64, P, P,
                                           P, i64, P, P, P, P]),
            "orc_bf16_round": (C.c_uint16, [f64]),
            "orc_sts_confidence": (f64, [f64, f64]),
            "orc_markov_draft_request": (C.c_int, [P, i64, P, P, i32, P, P, i32, i64, i32, u64,
                                                   u64, P, P, P, P, P, P]),
            "orc_schedule": (C.c_int, [P, P, i32, i32, P, i32, P, P, P, P]),
            "orc_schedule_rule": (C.c_int, [P, P, i32, i32, P, i32, i32, P, P, P, P]),
            "orc_schedule_async": (C.c_int, [P, i64, P, P, i32, i32, P, i32, i32, P, P, P, P]),
            "orc_acceptance_update": (C.c_int, [P, P, i32, i32, f64, f64, f64, P, P, P]),
            "orc_sts_fit": (C.c_int, [P, P, P, i32, i32, i32, f64, f64, i32, P, P, P, P, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _p(a):
    return None if a is None else a.ctypes.data


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _arr(a, dt):
    return None if a is None else np.ascontiguousarray(a, dtype=dt)


# ---- random numbers ------------------------------------------------------------------------

def philox4x32_10(ctr, key):
    c = np.asarray(ctr, dtype=np.uint32).copy()
    k = np.asarray(key, dtype=np.uint32).copy()
    out = np.zeros(4, dtype=np.uint32)
    _load().orc_philox4x32_10(c.ctypes.data, k.ctypes.data, out.ctypes.data)
    return out


def random_word(seed, req, pos, tag, v):
    return int(_load().orc_random_word(seed, req, pos, tag, v))


def uniform(seed, req, pos, tag, v):
    return float(_load().orc_uniform(seed, req, pos, tag, v))


def race_uniform(seed, req, pos, tag, v):
    return float(_load().orc_race_uniform(seed, req, pos, tag, v))


# ---- closed forms ----------------------------------------------------------------------------

def row_stats(row):
    row = _f32(row)
    M, S = C.c_double(), C.c_double()
    st = _load().orc_row_stats(row.ctypes.data, row.size, C.byref(M), C.byref(S))
    return st, M.value, S.value


def overlap(target_row, draft_row):
    t, d = _f32(target_row), _f32(draft_row)
    return float(_load().orc_overlap(t.ctypes.data, d.ctypes.data, t.size))


def expected_words(alpha, gamma):
    return float(_load().orc_expected_words(alpha, gamma))


def speedup(alpha, gamma, c):
    return float(_load().orc_speedup(alpha, gamma, c))


# ---- sampling --------------------------------------------------------------------------------

def sample_race(row, seed, req, pos, tag):
    row = _f32(row)
    tok, margin = C.c_int32(), C.c_double()
    st = _load().orc_sample_race(row.ctypes.data, row.size, seed, req, pos, tag, C.byref(tok),
                                 C.byref(margin))
    return st, tok.value, margin.value


def sample_draft_batch(draft, V, ld, draft_row0, draft_len, B, seed, request_ids=None,
                       n_draft_rows=None):
    draft = _f32(draft)
    draft_row0 = _arr(draft_row0, np.int64)
    draft_len = _arr(draft_len, np.int32)
    rids = _arr(request_ids, np.uint64)
    n = n_draft_rows if n_draft_rows is not None else draft.size // ld
    tokens = np.full(n, -1, dtype=np.int32)
    st = _load().orc_sample_draft_batch(draft.ctypes.data, V, ld, draft_row0.ctypes.data,
                                        draft_len.ctypes.data, B, seed, _p(rids),
                                        tokens.ctypes.data)
    return st, tokens


def lmhead_logits(hidden, W):
    """Logits of hidden [rows, H] through W [V, H]: binary64 sums rounded once to binary32."""
    hidden, W = _f32(hidden), _f32(W)
    rows, H = hidden.shape
    V = W.shape[0]
    out = np.zeros((rows, V), dtype=np.float32)
    st = _load().orc_lmhead_logits(hidden.ctypes.data, W.ctypes.data, rows, H, V, out.ctypes.data)
    assert st == OK
    return out


def race_shard(trow, drow, v_off, resid, w, stats, seed, req, pos, tag):
    """Best (key, global index) of the race over the vocabulary shard trow / drow (columns
    v_off ..), with the whole rows' statistics stats = (Mt, St, Md, Sd) (natural log)."""
    trow = _f32(trow)
    drow = _f32(drow) if drow is not None else trow
    key, idx = C.c_double(), C.c_int64()
    Mt, St, Md, Sd = (float(v) for v in stats)
    _load().orc_race_shard(trow.ctypes.data, drow.ctypes.data, trow.size, int(v_off), int(resid),
                           float(w), Mt, St, Md, Sd, seed, req, pos, tag, C.byref(key),
                           C.byref(idx))
    return key.value, idx.value


# ---- verification ----------------------------------------------------------------------------

def verify_token_request(target, draft, tokens, seed, req):
    target, draft = _f32(target), _f32(draft)
    tokens = _arr(tokens, np.int32)
    gamma = tokens.size
    V = target.shape[-1]
    ratio = np.zeros(max(gamma, 1))
    res = VerifyResult()
    _load().orc_verify_token_request(target.ctypes.data, draft.ctypes.data, V, V,
                                     tokens.ctypes.data, gamma, seed, req, ratio.ctypes.data,
                                     C.byref(res))
    return res, ratio[:gamma]


def verify_block_request(target, draft, tokens, seed, req):
    target, draft = _f32(target), _f32(draft)
    tokens = _arr(tokens, np.int32)
    gamma = tokens.size
    V = target.shape[-1]
    rho = np.zeros(max(gamma, 1))
    h = np.zeros(max(gamma, 1))
    res = VerifyResult()
    _load().orc_verify_block_request(target.ctypes.data, draft.ctypes.data, V, V,
                                     tokens.ctypes.data, gamma, seed, req, rho.ctypes.data,
                                     h.ctypes.data, C.byref(res))
    return res, rho[:gamma], h[:gamma]


def verify_batch(block, target, draft, V, ld, target_row0, draft_row0, draft_len, draft_tokens,
                 B, seed, request_ids=None, out_ld=None):
    """Batched verification laid out like the C-ABI calls; returns a dict of numpy outputs."""
    target, draft = _f32(target), _f32(draft)
    target_row0 = _arr(target_row0, np.int64)
    draft_row0 = _arr(draft_row0, np.int64)
    draft_len = _arr(draft_len, np.int32)
    draft_tokens = _arr(draft_tokens, np.int32)
    rids = _arr(request_ids, np.uint64)
    gmax = int(draft_len.max()) if B > 0 else 0
    out_ld = out_ld or gmax + 1
    acc = np.zeros(B, dtype=np.int32)
    out = np.zeros((B, out_ld), dtype=np.int32)
    corr = np.zeros(B, dtype=np.int32)
    ratio = np.full(draft_tokens.size, np.nan)
    h = np.full(draft_tokens.size, np.nan)
    results = (VerifyResult * max(B, 1))()
    st = _load().orc_verify_batch(int(block), target.ctypes.data, draft.ctypes.data, V, ld,
                                  target_row0.ctypes.data, draft_row0.ctypes.data,
                                  draft_len.ctypes.data, draft_tokens.ctypes.data, B, seed,
                                  _p(rids), acc.ctypes.data, out.ctypes.data, out_ld,
                                  corr.ctypes.data, ratio.ctypes.data, h.ctypes.data, results)
    res = list(results)[:B]
    return {
        "status": st,
        "accepted_len": acc,
        "out_tokens": out,
        "correction": corr,
        "ratio": ratio,
        "h": h,
        "race_kind": np.array([r.race_kind for r in res], dtype=np.int32),
        "req_status": np.array([r.status for r in res], dtype=np.int32),
        "decision_margin": np.array([r.decision_margin for r in res]),
        "race_margin": np.array([r.race_margin for r in res]),
    }


# ---- DSpark draft side ------------------------------------------------------------------------

def bf16_round(x):
    return int(_load().orc_bf16_round(float(x)))


def sts_confidence(s, T):
    return float(_load().orc_sts_confidence(float(s), float(T)))


def markov_draft_request(backbone, U, W, anchor, scores, T, seed, req, forced_prev=None,
                         want_z=True):
    """One request of the Markov-head draft.  backbone [K, V], U [V, R], W [R, V] (float32)."""
    backbone, U, W = _f32(backbone), _f32(U), _f32(W)
    scores, T = _f32(scores), _f32(T)
    K, V = backbone.shape
    R = U.shape[1]
    forced = _arr(forced_prev, np.int32)
    z = np.zeros((K, V), dtype=np.uint16) if want_z else None
    x = np.zeros(K, dtype=np.int32)
    stats = np.zeros((K, 2))
    conf = np.zeros(K)
    margin = np.zeros(K)
    st = _load().orc_markov_draft_request(backbone.ctypes.data, V, U.ctypes.data, W.ctypes.data,
                                          int(anchor), scores.ctypes.data, T.ctypes.data, K, V, R,
                                          seed, req, _p(forced), _p(z), x.ctypes.data,
                                          stats.ctypes.data, conf.ctypes.data, margin.ctypes.data)
    return {"status": st, "z": z, "x": x, "stats": stats, "conf": conf, "margin": margin}


STOP_FIRST_DROP = 0
STOP_ARGMAX = 1
STOP_FIXED_DEPTH = 2


def schedule(cond_accept, max_len, sps, B_max, rule=STOP_FIRST_DROP):
    c = _f32(cond_accept)
    N, K = c.shape
    ml = _arr(max_len, np.int32)
    sps = np.ascontiguousarray(sps, dtype=np.float64)
    sel = np.zeros(N, dtype=np.int32)
    surv = np.zeros((N, K), dtype=np.float32)
    total = C.c_int32()
    obj = C.c_double()
    st = _load().orc_schedule_rule(c.ctypes.data, ml.ctypes.data, N, K, sps.ctypes.data, B_max,
                                   int(rule), sel.ctypes.data, surv.ctypes.data, C.byref(total),
                                   C.byref(obj))
    return {"status": st, "sel_len": sel, "survival": surv, "total_rows": total.value,
            "objective": obj.value}


def schedule_async(conf_rounds, round_, prior, max_len, sps, B_max, rule=STOP_FIRST_DROP):
    """Round `round_` scheduled with the predictions of round `round_` - 2 (conf_rounds
    [rounds, N, K]; prior [N, K] for rounds 0 and 1)."""
    conf = _f32(conf_rounds)
    prior = _f32(prior)
    _, N, K = conf.shape
    ml = _arr(max_len, np.int32)
    sps = np.ascontiguousarray(sps, dtype=np.float64)
    sel = np.zeros(N, dtype=np.int32)
    surv = np.zeros((N, K), dtype=np.float32)
    total = C.c_int32()
    obj = C.c_double()
    st = _load().orc_schedule_async(conf.ctypes.data, int(round_), prior.ctypes.data,
                                    ml.ctypes.data, N, K, sps.ctypes.data, B_max, int(rule),
                                    sel.ctypes.data, surv.ctypes.data, C.byref(total),
                                    C.byref(obj))
    return {"status": st, "sel_len": sel, "survival": surv, "total_rows": total.value,
            "objective": obj.value}


def acceptance_update(sel_len, accepted_len, K, trials, accepts, decay=1.0, prior_a=1.0,
                      prior_b=1.0):
    """One round of the per-position acceptance counts (updated in place); returns (status,
    alpha float32 [K])."""
    sel = _arr(sel_len, np.int32)
    acc = _arr(accepted_len, np.int32)
    assert trials.dtype == np.float64 and accepts.dtype == np.float64
    assert trials.flags.c_contiguous and accepts.flags.c_contiguous
    alpha = np.zeros(K, dtype=np.float32)
    st = _load().orc_acceptance_update(sel.ctypes.data, acc.ctypes.data, sel.size, K,
                                       float(decay), float(prior_a), float(prior_b),
                                       trials.ctypes.data, accepts.ctypes.data, alpha.ctypes.data)
    return st, alpha


def sts_fit(scores, sel_len, accepted_len, iters=30, beta_min=1.0 / 16, beta_max=16.0, nbins=15):
    """Per-position temperatures fitted to the verified outcomes; returns a dict of per-position
    arrays (T, nll, ece_raw, ece_fit, count) and the status."""
    s = _f32(scores)
    N, K = s.shape
    sel = _arr(sel_len, np.int32)
    acc = _arr(accepted_len, np.int32)
    T = np.zeros(K, np.float32)
    nll, er, ef = np.zeros(K), np.zeros(K), np.zeros(K)
    cnt = np.zeros(K, np.int32)
    st = _load().orc_sts_fit(s.ctypes.data, sel.ctypes.data, acc.ctypes.data, N, K, int(iters),
                             float(beta_min), float(beta_max), int(nbins), T.ctypes.data,
                             nll.ctypes.data, er.ctypes.data, ef.ctypes.data, cnt.ctypes.data)
    return {"status": st, "T": T, "nll": nll, "ece_raw": er, "ece_fit": ef, "count": cnt}
