"""GB300 speculative-decoding verification: Python binding of ``libspecverify.so``.

The functions below carry the names of the C entry points declared in ``include/specverify.h`` and
do argument marshalling only: every step runs in the library's CUDA kernels.  Tensors must live on
the current CUDA device; outputs that are not supplied are allocated with torch.  The library is
loaded on first use and its absence raises -- there is no other implementation to fall back to.
"""
from __future__ import annotations

import ctypes as C
import os
import re
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libspecverify.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "specverify.h")

SV_OK, SV_ERR_INVALID, SV_ERR_UNSUPPORTED, SV_ERR_CUDA, SV_ERR_BAD_INPUT, SV_ERR_TIMEOUT = range(6)
SV_F32, SV_BF16 = 0, 1
SV_MAX_DRAFT_LEN = 64
SV_NOALLOC_SCRATCH_BYTES = 8 << 20  # scratch array of spec_verify_token_noalloc

_lock = threading.Lock()
_lib = None


class SpecVerifyError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        super().__init__(f"{where}: {status_string(code)}")


def declared_functions():
    """Names of the functions declared in include/specverify.h."""
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*"
                                 r"([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)))


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = C.CDLL(LIB_PATH)
        P, i32, i64, u64, sz = C.c_void_p, C.c_int32, C.c_int64, C.c_uint64, C.c_size_t
        st = C.c_int
        verify_args = [P, P, st, i64, i64, P, P, P, i32, P, i32, u64, P, P, P, i64, P]
        sigs = {
            "sv_status_string": (C.c_char_p, [st]),
            "sv_version": (C.c_char_p, []),
            "sv_profile_enable": (st, [C.c_int]),
            "sv_selftest_wait": (st, [i32, i32, P, P]),
            "sv_profile_read": (st, [P]),
            "spec_verify_workspace_bytes": (sz, [i32, i32, i64, st]),
            "spec_verify_token": (st, verify_args + [P, P, P, sz, P]),
            "spec_verify_block": (st, verify_args + [P, P, P, P, sz, P]),
            "spec_verify_token_noalloc": (st, verify_args + [P, P, P]),
            "spec_sample_draft": (st, [P, st, i64, i64, P, P, i32, i32, u64, P, P, P, P, sz, P]),
            "dspark_markov_workspace_bytes": (sz, [i32, i32, i64, i32]),
            "dspark_markov_draft": (st, [P, i64, P, P, i64, P, P, P, i32, i32, i64, i32, u64, P,
                                         P, P, i64, P, P, P, P, sz, P]),
            "dspark_schedule_workspace_bytes": (sz, [i32, i32]),
            "dspark_schedule": (st, [P, P, i32, i32, P, i32, P, P, P, P, P, P, sz, P]),
            "spec_verify_shard_stats": (st, [P, P, st, i64, i64, i64, i64, P, P, P, i32, P, i32,
                                             P, P, P, P, sz, P]),
            "spec_verify_shard_merge": (st, [P, P, i32, i64, P, P, P]),
            "spec_verify_shard_race": (st, [P, P, st, i64, i64, i64, i64, P, P, P, i32, P, i32,
                                            u64, P, P, P, P, P, P, P, P, sz, P]),
            "spec_verify_shard_finish": (st, [P, i32, i32, P, P, P, P, i64, P, P, P]),
            "spec_verify_lmhead_workspace_bytes": (sz, [i32, i32, i64, i64]),
            "spec_verify_lmhead": (st, [P, P, i64, P, i64, i64, i64, P, P, P, i32, P, i32, u64,
                                        P, P, P, i64, P, P, P, P, P, sz, P]),
            "dspark_schedule_rule": (st, [P, P, i32, i32, P, i32, i32, P, P, P, P, P, P, sz, P]),
            "dspark_schedule_async": (st, [P, i32, i64, P, P, i32, i32, P, i32, i32, P, P, P, P, P,
                                           P, sz, P]),
            "dspark_acceptance_update": (st, [P, P, i32, i32, C.c_double, C.c_double, C.c_double,
                                              P, P, P, P, P, P]),
            "dspark_sts_fit": (st, [P, P, P, i32, i32, i32, C.c_double, C.c_double, i32, P, P, P,
                                    P, P, P, P]),
        }
        for name, (res, args) in sigs.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
        return L


def status_string(code):
    return lib().sv_status_string(int(code)).decode()


def version():
    return lib().sv_version().decode()


def sv_selftest_wait(which, limit_us, status, stream=None):
    """Make one of the kernels' bounded waits run out (see include/specverify.h)."""
    _check(lib().sv_selftest_wait(int(which), int(limit_us), _ptr(status), _stream(stream)),
           "sv_selftest_wait")


def sv_profile_enable(enable=True):
    _check(lib().sv_profile_enable(int(enable)), "sv_profile_enable")


def sv_profile_read():
    """Durations (ms) of the last profiled verify call: [streaming, decisions, race]."""
    out = (C.c_float * 3)()
    _check(lib().sv_profile_read(out), "sv_profile_read")
    return [float(x) for x in out]


def _check(code, where):
    if code != SV_OK:
        raise SpecVerifyError(code, where)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _dtype_code(t):
    if t.dtype == torch.bfloat16:
        return SV_BF16
    if t.dtype == torch.float32:
        return SV_F32
    raise TypeError(f"logits must be bfloat16 or float32, got {t.dtype}")


def _dev(t, dtype=None, rows=False, strided=False):
    """Checks a device tensor; `rows` allows a row-strided 2-D view (logits with ld > V) and
    `strided` leaves the layout to the caller's own checks."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors passed to the library must be on a CUDA device")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"expected {dtype}, got {t.dtype}")
    if rows:
        if t.dim() != 2 or t.stride(1) != 1:
            raise ValueError("logits must be a 2-D tensor with unit column stride")
    elif not strided and not t.is_contiguous():
        raise ValueError("tensors passed to the library must be contiguous")
    return t


_ws_cache = {}


def workspace(nbytes, device=None):
    """A cached device buffer of at least `nbytes` bytes (256-byte aligned, from torch)."""
    device = torch.device(device or torch.cuda.current_device())
    key = (device.index, threading.get_ident())
    buf = _ws_cache.get(key)
    if buf is None or buf.numel() < nbytes:
        buf = torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)
        _ws_cache[key] = buf
    return buf


# ---- verification ----------------------------------------------------------------------------

def spec_verify_workspace_bytes(B, max_draft_len, V, dtype_code):
    return int(lib().spec_verify_workspace_bytes(B, max_draft_len, V, dtype_code))


def _verify(block, target, draft, target_row0, draft_row0, draft_len, max_draft_len,
            draft_tokens, seed, request_ids, out_ld, want_rows, status, ws, stream):
    _dev(target, rows=True), _dev(draft, rows=True)
    _dev(target_row0, torch.int64), _dev(draft_row0, torch.int64)
    _dev(draft_len, torch.int32), _dev(draft_tokens, torch.int32)
    _dev(request_ids)
    dt = _dtype_code(target)
    if draft.dtype != target.dtype:
        raise TypeError("target and draft logits must have the same dtype")
    V = target.shape[-1]
    ld = target.stride(0)
    if draft.stride(0) != ld:
        raise ValueError("target and draft rows must have the same stride")
    B = draft_len.numel()
    out_ld = out_ld or max_draft_len + 1
    dev = target.device
    accepted = torch.empty(B, dtype=torch.int32, device=dev)
    out_tokens = torch.empty((B, out_ld), dtype=torch.int32, device=dev)
    correction = torch.empty(B, dtype=torch.int32, device=dev)
    n_draft_rows = draft_tokens.numel()
    rows_a = torch.empty(n_draft_rows, dtype=torch.float32, device=dev) if want_rows else None
    rows_h = (torch.empty(n_draft_rows, dtype=torch.float32, device=dev)
              if (want_rows and block) else None)
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=dev)
    need = spec_verify_workspace_bytes(B, max_draft_len, V, dt)
    if ws is None:
        ws = workspace(need, dev)
    args = [_ptr(target), _ptr(draft), dt, V, ld, _ptr(target_row0), _ptr(draft_row0),
            _ptr(draft_len), int(max_draft_len), _ptr(draft_tokens), B, int(seed),
            _ptr(request_ids), _ptr(accepted), _ptr(out_tokens), out_ld, _ptr(correction)]
    if block:
        code = lib().spec_verify_block(*args, _ptr(rows_a), _ptr(rows_h), _ptr(status),
                                       _ptr(ws), ws.numel(), _stream(stream))
    else:
        code = lib().spec_verify_token(*args, _ptr(rows_a), _ptr(status), _ptr(ws), ws.numel(),
                                       _stream(stream))
    _check(code, "spec_verify_block" if block else "spec_verify_token")
    out = {"accepted_len": accepted, "out_tokens": out_tokens, "correction": correction,
           "status": status}
    if block:
        out["running_ratio"] = rows_a
        out["h"] = rows_h
    else:
        out["accept_ratio"] = rows_a
    return out


def spec_verify_token(target, draft, target_row0, draft_row0, draft_len, max_draft_len,
                      draft_tokens, seed, request_ids=None, out_ld=None, want_ratio=True,
                      status=None, workspace=None, stream=None):
    """Token-level verification (see include/specverify.h).  Returns a dict of device tensors."""
    return _verify(False, target, draft, target_row0, draft_row0, draft_len, max_draft_len,
                   draft_tokens, seed, request_ids, out_ld, want_ratio, status, workspace, stream)


def spec_verify_block(target, draft, target_row0, draft_row0, draft_len, max_draft_len,
                      draft_tokens, seed, request_ids=None, out_ld=None, want_rows=True,
                      status=None, workspace=None, stream=None):
    """Block verification (see include/specverify.h).  Returns a dict of device tensors."""
    return _verify(True, target, draft, target_row0, draft_row0, draft_len, max_draft_len,
                   draft_tokens, seed, request_ids, out_ld, want_rows, status, workspace, stream)


def spec_verify_lmhead_workspace_bytes(B, max_draft_len, V, H):
    return int(lib().spec_verify_lmhead_workspace_bytes(B, max_draft_len, V, H))


def spec_verify_lmhead(target_hidden, draft_hidden, W, target_row0, draft_row0, draft_len,
                       max_draft_len, draft_tokens, seed, request_ids=None, out_ld=None,
                       want_ratio=True, status=None, workspace=None, stream=None):
    """Token-level verification from hidden states: logits = hidden rows x W^T (bf16 operands,
    W [V, H]), decided and sampled as spec_verify_token does (see include/specverify.h).
    Returns a dict of device tensors."""
    _dev(target_hidden, torch.bfloat16, rows=True), _dev(draft_hidden, torch.bfloat16, rows=True)
    _dev(W, torch.bfloat16, rows=True)
    _dev(target_row0, torch.int64), _dev(draft_row0, torch.int64)
    _dev(draft_len, torch.int32), _dev(draft_tokens, torch.int32)
    _dev(request_ids)
    H = target_hidden.shape[-1]
    if draft_hidden.shape[-1] != H or W.shape[-1] != H:
        raise ValueError("hidden rows and W must have the same width H")
    ldh = target_hidden.stride(0)
    if draft_hidden.stride(0) != ldh:
        raise ValueError("target and draft hidden rows must have the same stride")
    V = W.shape[0]
    B = draft_len.numel()
    out_ld = out_ld or max_draft_len + 1
    dev = target_hidden.device
    accepted = torch.empty(B, dtype=torch.int32, device=dev)
    out_tokens = torch.empty((B, out_ld), dtype=torch.int32, device=dev)
    correction = torch.empty(B, dtype=torch.int32, device=dev)
    ratio = (torch.empty(draft_tokens.numel(), dtype=torch.float32, device=dev)
             if want_ratio else None)
    recomputed = torch.zeros(1, dtype=torch.int32, device=dev)
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=dev)
    need = spec_verify_lmhead_workspace_bytes(B, max_draft_len, V, H)
    ws = workspace if workspace is not None else globals()["workspace"](need, dev)
    code = lib().spec_verify_lmhead(_ptr(target_hidden), _ptr(draft_hidden), ldh, _ptr(W),
                                    W.stride(0), H, V, _ptr(target_row0), _ptr(draft_row0),
                                    _ptr(draft_len), int(max_draft_len), _ptr(draft_tokens), B,
                                    int(seed), _ptr(request_ids), _ptr(accepted),
                                    _ptr(out_tokens), out_ld, _ptr(correction), _ptr(ratio),
                                    _ptr(recomputed), _ptr(status), _ptr(ws), ws.numel(),
                                    _stream(stream))
    _check(code, "spec_verify_lmhead")
    return {"accepted_len": accepted, "out_tokens": out_tokens, "correction": correction,
            "accept_ratio": ratio, "recomputed": recomputed, "status": status}


def spec_sample_draft(draft, draft_row0, draft_len, max_draft_len, seed, request_ids=None,
                      draft_tokens=None, status=None, workspace=None, stream=None):
    """Sample draft tokens from q for every drafted row; returns the token tensor (by draft row)."""
    _dev(draft, rows=True), _dev(draft_row0, torch.int64), _dev(draft_len, torch.int32)
    dt = _dtype_code(draft)
    V = draft.shape[-1]
    ld = draft.stride(0)
    B = draft_len.numel()
    dev = draft.device
    if draft_tokens is None:
        draft_tokens = torch.full((draft.shape[0],), -1, dtype=torch.int32, device=dev)
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=dev)
    need = spec_verify_workspace_bytes(B, max_draft_len, V, dt)
    ws = workspace if workspace is not None else globals()["workspace"](need, dev)
    code = lib().spec_sample_draft(_ptr(draft), dt, V, ld, _ptr(draft_row0), _ptr(draft_len),
                                   int(max_draft_len), B, int(seed), _ptr(request_ids),
                                   _ptr(draft_tokens), _ptr(status), _ptr(ws), ws.numel(),
                                   _stream(stream))
    _check(code, "spec_sample_draft")
    return draft_tokens


# ---- vocabulary-sharded verification ------------------------------------------------------------

def spec_verify_shard_stats(target, draft, v_off, V_total, target_row0, draft_row0, draft_len,
                            max_draft_len, draft_tokens, status=None, workspace=None, stream=None):
    """This shard's statistics of every drafted row pair and the drafted tokens' logits (-inf
    where the shard does not hold the token).  Returns (stats fp32 [B * gmax, 4], tok fp32
    [B * gmax, 2])."""
    _dev(target, rows=True), _dev(draft, rows=True)
    _dev(target_row0, torch.int64), _dev(draft_row0, torch.int64)
    _dev(draft_len, torch.int32), _dev(draft_tokens, torch.int32)
    dt = _dtype_code(target)
    Vs, ld = target.shape[-1], target.stride(0)
    B = draft_len.numel()
    dev = target.device
    units = max(1, B * max_draft_len)
    stats = torch.empty((units, 4), dtype=torch.float32, device=dev)
    tok = torch.empty((units, 2), dtype=torch.float32, device=dev)
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=dev)
    need = spec_verify_workspace_bytes(B, max_draft_len, Vs, dt)
    ws = workspace if workspace is not None else globals()["workspace"](need, dev)
    code = lib().spec_verify_shard_stats(_ptr(target), _ptr(draft), dt, Vs, ld, int(v_off),
                                         int(V_total), _ptr(target_row0), _ptr(draft_row0),
                                         _ptr(draft_len), int(max_draft_len), _ptr(draft_tokens),
                                         B, _ptr(stats), _ptr(tok), _ptr(status), _ptr(ws),
                                         ws.numel(), _stream(stream))
    _check(code, "spec_verify_shard_stats")
    return stats, tok


def spec_verify_shard_merge(stats_all, tok_all, stream=None):
    """Statistics of every shard ([n, rows, 4]) merged in shard order; drafted-token logits
    ([n, rows, 2]) from the shard that holds each token."""
    _dev(stats_all, torch.float32), _dev(tok_all, torch.float32)
    n, rows = stats_all.shape[0], stats_all.shape[1]
    stats = torch.empty((rows, 4), dtype=torch.float32, device=stats_all.device)
    tok = torch.empty((rows, 2), dtype=torch.float32, device=stats_all.device)
    code = lib().spec_verify_shard_merge(_ptr(stats_all.contiguous()), _ptr(tok_all.contiguous()),
                                         n, rows, _ptr(stats), _ptr(tok), _stream(stream))
    _check(code, "spec_verify_shard_merge")
    return stats, tok


def spec_verify_shard_race(target, draft, v_off, V_total, target_row0, draft_row0, draft_len,
                           max_draft_len, draft_tokens, seed, stats, tok, request_ids=None,
                           want_ratio=True, status=None, workspace=None, stream=None):
    """Every request decided from the merged statistics, then this shard's race.  Returns
    {"accepted_len", "winners" (int64 [B, 2], unsigned bit patterns), "accept_ratio", "status"}."""
    _dev(target, rows=True), _dev(draft, rows=True), _dev(request_ids)
    dt = _dtype_code(target)
    Vs, ld = target.shape[-1], target.stride(0)
    B = draft_len.numel()
    dev = target.device
    acc = torch.empty(B, dtype=torch.int32, device=dev)
    winners = torch.empty((B, 2), dtype=torch.int64, device=dev)
    ratio = (torch.empty(draft_tokens.numel(), dtype=torch.float32, device=dev)
             if want_ratio else None)
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=dev)
    need = spec_verify_workspace_bytes(B, max_draft_len, Vs, dt)
    ws = workspace if workspace is not None else globals()["workspace"](need, dev)
    code = lib().spec_verify_shard_race(_ptr(target), _ptr(draft), dt, Vs, ld, int(v_off),
                                        int(V_total), _ptr(target_row0), _ptr(draft_row0),
                                        _ptr(draft_len), int(max_draft_len), _ptr(draft_tokens),
                                        B, int(seed), _ptr(request_ids), _ptr(stats), _ptr(tok),
                                        _ptr(acc), _ptr(ratio), _ptr(winners), _ptr(status),
                                        _ptr(ws), ws.numel(), _stream(stream))
    _check(code, "spec_verify_shard_race")
    return {"accepted_len": acc, "winners": winners, "accept_ratio": ratio, "status": status}


def spec_verify_shard_finish(winners_all, accepted_len, draft_row0, draft_tokens, out_ld,
                             status=None, stream=None):
    """The largest winner over the shards ([n, B, 2]) and the request outputs."""
    _dev(winners_all, torch.int64), _dev(accepted_len, torch.int32)
    n, B = winners_all.shape[0], winners_all.shape[1]
    dev = winners_all.device
    out = torch.empty((B, out_ld), dtype=torch.int32, device=dev)
    corr = torch.empty(B, dtype=torch.int32, device=dev)
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=dev)
    code = lib().spec_verify_shard_finish(_ptr(winners_all.contiguous()), n, B,
                                          _ptr(accepted_len), _ptr(draft_row0),
                                          _ptr(draft_tokens), _ptr(out), int(out_ld),
                                          _ptr(corr), _ptr(status), _stream(stream))
    _check(code, "spec_verify_shard_finish")
    return {"out_tokens": out, "correction": corr, "accepted_len": accepted_len,
            "status": status}


def all_gather_stacked(t, group=None):
    """The tensor t of every rank of `group`, stacked in rank order (the shard order)."""
    import torch.distributed as dist
    parts = [torch.empty_like(t) for _ in range(dist.get_world_size(group))]
    dist.all_gather(parts, t.contiguous(), group=group)
    return torch.stack(parts)


def spec_verify_token_sharded(target, draft, v_off, V_total, target_row0, draft_row0, draft_len,
                              max_draft_len, draft_tokens, seed, request_ids=None, out_ld=None,
                              gather=all_gather_stacked, steps=None):
    """Token-level verification of this rank's vocabulary shard (columns v_off .. v_off + Vs of
    every row), rank r holding shard r: the four library calls with the two exchanges between
    them, `gather(t)` stacking every rank's t in rank order (all_gather over the default process
    group by default).  `steps` replaces the four calls (a dict with keys stats, merge, race,
    finish taking the same arguments) -- the exchanges stay the same."""
    st = steps or {"stats": spec_verify_shard_stats, "merge": spec_verify_shard_merge,
                   "race": spec_verify_shard_race, "finish": spec_verify_shard_finish}
    stats, tok = st["stats"](target, draft, v_off, V_total, target_row0, draft_row0, draft_len,
                             max_draft_len, draft_tokens)
    stats, tok = st["merge"](gather(stats), gather(tok))
    race = st["race"](target, draft, v_off, V_total, target_row0, draft_row0, draft_len,
                      max_draft_len, draft_tokens, seed, stats, tok, request_ids=request_ids)
    out = st["finish"](gather(race["winners"]), race["accepted_len"], draft_row0, draft_tokens,
                       out_ld or max_draft_len + 1)
    out["accept_ratio"] = race.get("accept_ratio")
    return out


# ---- DSpark draft side ------------------------------------------------------------------------

def dspark_markov_workspace_bytes(B, K, V, R):
    return int(lib().dspark_markov_workspace_bytes(B, K, V, R))


def dspark_markov_draft(backbone, U, Wt, anchor, conf_scores, sts_T, seed, request_ids=None,
                        want_logits=True, want_stats=True, status=None, workspace=None,
                        stream=None):
    """Markov-head drafting.  backbone bf16 [B, K, V] (rows may be padded: stride(1) = ldb,
    stride(0) = K * ldb); U bf16 [V, R]; Wt bf16 [V, R] (W stored transposed, rows may be padded);
    anchor int32 [B]; conf_scores fp32 [B, K] and sts_T fp32 [K], or both None (no confidence)."""
    _dev(backbone, torch.bfloat16, strided=True), _dev(U, torch.bfloat16)
    _dev(Wt, torch.bfloat16, strided=True), _dev(anchor, torch.int32)
    if conf_scores is not None:
        _dev(conf_scores, torch.float32), _dev(sts_T, torch.float32)
    B, K, V = backbone.shape
    R = U.shape[1]
    ldb = backbone.stride(1)
    if backbone.stride(2) != 1 or backbone.stride(0) != K * ldb:
        raise ValueError("backbone must be [B, K, V] with unit column stride and rows ldb apart")
    if U.stride(1) != 1 or U.stride(0) != R or Wt.stride(1) != 1 or Wt.shape[0] != V:
        raise ValueError("U must be a contiguous [V, R] tensor and Wt a [V, R] row-major tensor")
    dev = backbone.device
    tokens = torch.empty((B, K), dtype=torch.int32, device=dev)
    ldz = (V + 7) // 8 * 8  # rows of z start on 16-byte boundaries
    z = (torch.empty((B, K, ldz), dtype=torch.bfloat16, device=dev)[:, :, :V] if want_logits
         else None)
    stats = torch.empty((B, K, 2), dtype=torch.float32, device=dev) if want_stats else None
    conf = torch.empty((B, K), dtype=torch.float32, device=dev) if conf_scores is not None else None
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=dev)
    need = dspark_markov_workspace_bytes(B, K, V, R)
    ws = workspace if workspace is not None else globals()["workspace"](need, dev)
    code = lib().dspark_markov_draft(_ptr(backbone), ldb, _ptr(U), _ptr(Wt), Wt.stride(0),
                                     _ptr(anchor), _ptr(conf_scores), _ptr(sts_T), B, K, V, R,
                                     int(seed), _ptr(request_ids), _ptr(tokens), _ptr(z),
                                     ldz, _ptr(stats), _ptr(conf), _ptr(status), _ptr(ws),
                                     ws.numel(), _stream(stream))
    _check(code, "dspark_markov_draft")
    return {"draft_tokens": tokens, "draft_logits": z, "row_stats": stats, "conf": conf,
            "status": status}


def dspark_schedule_workspace_bytes(N, K):
    return int(lib().dspark_schedule_workspace_bytes(N, K))


SV_STOP_FIRST_DROP = 0
SV_STOP_ARGMAX = 1
SV_STOP_FIXED_DEPTH = 2


def dspark_schedule(cond_accept, max_len, sps, B_max, want_survival=True, status=None,
                    workspace=None, stream=None, rule=SV_STOP_FIRST_DROP):
    """Hardware-aware prefix scheduler.  cond_accept fp32 [N, K]; sps fp64 [B_max + 1]; rule:
    SV_STOP_FIRST_DROP (early stop), SV_STOP_ARGMAX (best budget over all) or
    SV_STOP_FIXED_DEPTH (one depth for every request)."""
    _dev(cond_accept, torch.float32), _dev(max_len, torch.int32), _dev(sps, torch.float64)
    N, K = cond_accept.shape
    dev = cond_accept.device
    sel = torch.empty(N, dtype=torch.int32, device=dev)
    surv = torch.empty((N, K), dtype=torch.float32, device=dev) if want_survival else None
    total = torch.empty(1, dtype=torch.int32, device=dev)
    obj = torch.empty(1, dtype=torch.float64, device=dev)
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=dev)
    need = dspark_schedule_workspace_bytes(N, K)
    ws = workspace if workspace is not None else globals()["workspace"](need, dev)
    code = lib().dspark_schedule_rule(_ptr(cond_accept), _ptr(max_len), N, K, _ptr(sps),
                                      int(B_max), int(rule), _ptr(sel), _ptr(surv), _ptr(total),
                                      _ptr(obj), _ptr(status), _ptr(ws), ws.numel(),
                                      _stream(stream))
    _check(code, "dspark_schedule_rule")
    return {"sel_len": sel, "survival": surv, "total_rows": total, "objective": obj,
            "status": status}


def dspark_schedule_async(conf_ring, round_, cond_prior, max_len, sps, B_max, rule=SV_STOP_FIRST_DROP,
                          want_survival=True, status=None, workspace=None, stream=None):
    """Round `round_` scheduled with the confidences of round `round_` - 2: conf_ring fp32
    [depth >= 3, N, K] (round t's confidence head writes slot t % depth), cond_prior fp32 [N, K] for
    the first two rounds; otherwise as dspark_schedule."""
    _dev(conf_ring, torch.float32), _dev(cond_prior, torch.float32)
    _dev(max_len, torch.int32), _dev(sps, torch.float64)
    depth, N, K = conf_ring.shape
    if tuple(cond_prior.shape) != (N, K):
        raise ValueError("cond_prior must be [N, K] like one ring slot")
    dev = conf_ring.device
    sel = torch.empty(N, dtype=torch.int32, device=dev)
    surv = torch.empty((N, K), dtype=torch.float32, device=dev) if want_survival else None
    total = torch.empty(1, dtype=torch.int32, device=dev)
    obj = torch.empty(1, dtype=torch.float64, device=dev)
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=dev)
    need = dspark_schedule_workspace_bytes(N, K)
    ws = workspace if workspace is not None else globals()["workspace"](need, dev)
    code = lib().dspark_schedule_async(_ptr(conf_ring), int(depth), int(round_), _ptr(cond_prior),
                                       _ptr(max_len), N, K, _ptr(sps), int(B_max), int(rule),
                                       _ptr(sel), _ptr(surv), _ptr(total), _ptr(obj),
                                       _ptr(status), _ptr(ws), ws.numel(), _stream(stream))
    _check(code, "dspark_schedule_async")
    return {"sel_len": sel, "survival": surv, "total_rows": total, "objective": obj,
            "status": status}


def dspark_acceptance_update(sel_len, accepted_len, trials, accepts, decay=1.0, prior_a=1.0,
                             prior_b=1.0, alpha=None, cond_accept_out=None, status=None,
                             stream=None):
    """One verified round into the per-position acceptance counts (fp64 [K] device tensors,
    updated in place).  Returns {"alpha": fp32 [K], "cond_accept": fp32 [N, K] or None,
    "status"}."""
    _dev(sel_len, torch.int32), _dev(accepted_len, torch.int32)
    _dev(trials, torch.float64), _dev(accepts, torch.float64)
    N = sel_len.numel()
    K = trials.numel()
    if accepts.numel() != K or accepted_len.numel() != N:
        raise ValueError("inconsistent sizes")
    dev = trials.device
    if alpha is None:
        alpha = torch.empty(K, dtype=torch.float32, device=dev)
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=dev)
    code = lib().dspark_acceptance_update(_ptr(sel_len), _ptr(accepted_len), N, K, float(decay),
                                          float(prior_a), float(prior_b), _ptr(trials),
                                          _ptr(accepts), _ptr(alpha), _ptr(cond_accept_out),
                                          _ptr(status), _stream(stream))
    _check(code, "dspark_acceptance_update")
    return {"alpha": alpha, "cond_accept": cond_accept_out, "status": status}


def dspark_sts_fit(scores, sel_len, accepted_len, iters=30, beta_min=1.0 / 16, beta_max=16.0,
                   nbins=15, status=None, stream=None):
    """Per-position temperatures of the confidence head fitted to verified outcomes (scores fp32
    [N, K], sel_len / accepted_len int32 [N], all on the device).  Returns device tensors T [K],
    nll, ece_raw, ece_fit (fp64 [K]), count (int32 [K]) and status."""
    _dev(scores, torch.float32), _dev(sel_len, torch.int32), _dev(accepted_len, torch.int32)
    N, K = scores.shape
    dev = scores.device
    out = {"T": torch.empty(K, dtype=torch.float32, device=dev),
           "nll": torch.empty(K, dtype=torch.float64, device=dev),
           "ece_raw": torch.empty(K, dtype=torch.float64, device=dev),
           "ece_fit": torch.empty(K, dtype=torch.float64, device=dev),
           "count": torch.empty(K, dtype=torch.int32, device=dev),
           "status": status if status is not None else torch.zeros(1, dtype=torch.int32,
                                                                   device=dev)}
    code = lib().dspark_sts_fit(_ptr(scores), _ptr(sel_len), _ptr(accepted_len), N, K,
                                int(iters), float(beta_min), float(beta_max), int(nbins),
                                _ptr(out["T"]), _ptr(out["nll"]), _ptr(out["ece_raw"]),
                                _ptr(out["ece_fit"]), _ptr(out["count"]), _ptr(out["status"]),
                                _stream(stream))
    _check(code, "dspark_sts_fit")
    return out
