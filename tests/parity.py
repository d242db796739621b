"""GPU <-> oracle comparison helpers for the parity tests.

Policy: accepted lengths, emitted tokens and scheduler selections are compared bit for bit, except
requests whose oracle decision margin |u - threshold| or race margin (best minus second-best key)
is below 1e-5 -- those are counted and reported, never silently passed, and at most 1% of the
requests (at least one) may differ on them.  Probabilities (ratios, running ratios, thresholds)
must agree within 1e-5 relative.
"""
import numpy as np
import torch

NEAR_TIE = 1e-5
REL_TOL = 1e-5
EXEMPT_FRAC = 0.01  # largest share of requests that may differ on exempt (near-tie) decisions
RHO_PREC = 2e-6  # relative precision of a binary32 running ratio built from fp32 row sums
# absolute precision of a binary32 residual mass R: every term max(rho p - q, 0) carries the
# rounding of its two exponentials and of one fma (about 3 * 2^-22 of rho p), and the terms of rho p
# add up to at most rho <= 1, so |dR| < 7.2e-7 plus the summation's rounding
R_ABS = 1e-6


def host_f32(t):
    """Device logits -> float32 numpy rows (bf16 widens exactly)."""
    return t.float().cpu().numpy()


def layout_np(inp):
    return {k: inp[k].cpu().numpy() if torch.is_tensor(inp[k]) else inp[k]
            for k in ("target_row0", "draft_row0", "draft_len")}


def oracle_tokens(orc, inp, n_draft_rows=None):
    """Draft tokens sampled from q by the oracle (inputs for both sides)."""
    lay = layout_np(inp)
    draft = host_f32(inp["draft"])
    st, toks = orc.sample_draft_batch(draft, inp["V"], draft.shape[1], lay["draft_row0"],
                                      lay["draft_len"], inp["B"], inp["seed"],
                                      n_draft_rows=n_draft_rows)
    assert st == 0
    return toks


def oracle_verify(orc, block, inp, tokens, request_ids=None):
    lay = layout_np(inp)
    tgt = host_f32(inp["target"])
    drf = host_f32(inp["draft"])
    return orc.verify_batch(block, tgt, drf, inp["V"], tgt.shape[1], lay["target_row0"],
                            lay["draft_row0"], lay["draft_len"], tokens, inp["B"], inp["seed"],
                            request_ids=request_ids, out_ld=inp["max_draft_len"] + 1)


def _rel_err(a, b, floor=1e-30):
    return np.abs(a - b) / np.maximum(np.abs(b), floor)


def compare_verify(gpu, ref, block, lens, draft_row0, report=None, near_tie=NEAR_TIE,
                   rel_tol=REL_TOL):
    """Asserts parity; returns counts {requests, exempt, exempt_mismatch}.  `near_tie` and
    `rel_tol` replace the margins and the ratio tolerance where the two sides' logits themselves
    differ by rounding (logits computed from hidden states)."""
    acc = gpu["accepted_len"].cpu().numpy()
    out = gpu["out_tokens"].cpu().numpy()
    exempt = (ref["decision_margin"] < near_tie) | (ref["race_margin"] < near_tie)
    mism = (acc != ref["accepted_len"]) | np.any(out != ref["out_tokens"], axis=1)
    bad = mism & ~exempt
    assert not bad.any(), (
        f"{bad.sum()} requests differ: idx {np.flatnonzero(bad)[:8]}, gpu acc "
        f"{acc[bad][:8]}, ref acc {ref['accepted_len'][bad][:8]}, gpu tok "
        f"{out[bad][:4]}, ref tok {ref['out_tokens'][bad][:4]}")
    # per-position probabilities of every drafted row
    rows = np.concatenate([np.arange(r0, r0 + g) for r0, g in zip(draft_row0, lens)]).astype(
        np.int64) if len(lens) else np.zeros(0, np.int64)
    row_out = gpu.get("running_ratio" if block else "accept_ratio")
    if row_out is None:  # the call left out its per-row outputs
        rows = rows[:0]
    if rows.size:
        if block:
            g_rho = gpu["running_ratio"].cpu().numpy()[rows]
            g_h = gpu["h"].cpu().numpy()[rows]
            r_rho = ref["ratio"][rows]
            r_h = ref["h"][rows]
            assert np.all(_rel_err(g_rho, r_rho, 1e-6) < REL_TOL)
            # h = R / (R + 1 - rho) is ill-conditioned when R + 1 - rho is small.  With
            # R + 1 - rho = R / h and R = h (1 - rho) / (1 - h), first-order propagation of an
            # absolute error dR of the residual mass and a relative error drho of rho gives
            #   |dh| <= [(1 - h)^2 dR + h (1 - h) rho drho] / (1 - rho);
            # binary32 sums give dR <= R_ABS and drho <= RHO_PREC.
            one_h = np.maximum(1 - r_h, 0)
            cond = ((one_h ** 2) * R_ABS + r_h * one_h * r_rho * RHO_PREC) / np.maximum(
                1 - r_rho, 1e-30)
            tol = REL_TOL * np.abs(r_h) + cond
            err = np.abs(g_h - r_h)
            assert np.all(err <= tol), (np.max(err / tol), np.max(err))
            extra = {"max_rel_err_rho": float(np.max(_rel_err(g_rho, r_rho, 1e-6))),
                     "max_h_err_over_tol": float(np.max(err / np.maximum(tol, 1e-30)))}
        else:
            g_a = gpu["accept_ratio"].cpu().numpy()[rows]
            rel = _rel_err(g_a, ref["ratio"][rows], 1e-6)
            assert np.all(rel < rel_tol), np.max(rel)
            extra = {"max_rel_err_ratio": float(np.max(rel))}
    res = {"requests": int(acc.size), "exempt": int(exempt.sum()),
           "exempt_mismatch": int((mism & exempt).sum())}
    # near ties may decide either way, but only a few of them can: more than 1% of the requests
    # (at least one) differing on exempt decisions points at a systematic error, not at rounding
    assert res["exempt_mismatch"] <= max(1, int(np.ceil(EXEMPT_FRAC * acc.size))), res
    if rows.size:
        res.update(extra)
    if report is not None:
        report.append(res)
    return res
