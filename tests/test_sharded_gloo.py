"""Vocabulary-sharded verification across ranks, on the CPU: two gloo ranks each hold one shard
of every logit row (the vocabulary split at a multiple of 8) and run the library's orchestration
(spec_verify_token_sharded: its exchanges are real all-gathers over the process group) with the
four per-shard steps restated from the oracle -- per-shard softmax statistics, their log-sum-exp
merge, the decision and the race over the shard keyed by global vocabulary indices, the largest
winner.  The result must equal the oracle's verification of the unsharded rows.  This pins the
decomposition the GPU shard kernels implement and the exchange order; the kernels themselves are
compared with the oracle on one GPU (test_gpu_shard.py)."""
import math
import os
import socket
import sys

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
B, G, V, SPLIT, SEED = 10, 4, 3000, 1504, 7


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs():
    sys.path.insert(0, ROOT)
    from speculative_decoding_verification_token_gb300 import synth
    w = synth.scaled(synth.TOKEN_LARGE, B=B, gamma=G, V=V, dtype=torch.float32, draft_noise=0.7)
    inp = synth.token_inputs(w, device="cpu", draft_len=synth.ragged_lengths(B, G, seed=3))
    return w, inp


def _oracle_steps(orc, t_rows, d_rows, lay, tokens):
    """The four steps restated from the oracle (natural-log statistics, float64)."""
    def stats(target, draft, v_off, V_total, target_row0, draft_row0, draft_len, gmax, toks):
        st = np.zeros((B * gmax, 4))
        tk = np.full((B * gmax, 2), -np.inf)
        for r in range(B):
            for i in range(1, int(lay["draft_len"][r]) + 1):
                u = r * gmax + i - 1
                trow = target[int(lay["target_row0"][r]) + i - 1]
                drow = draft[int(lay["draft_row0"][r]) + i - 1]
                _, st[u, 0], st[u, 1] = orc.row_stats(trow)
                _, st[u, 2], st[u, 3] = orc.row_stats(drow)
                x = int(toks[int(lay["draft_row0"][r]) + i - 1]) - v_off
                if 0 <= x < trow.size:
                    tk[u] = (trow[x], drow[x])
        return torch.from_numpy(st), torch.from_numpy(tk)

    def merge(stats_all, tok_all):
        s = stats_all.numpy()
        m_t, m_d = s[:, :, 0].max(0), s[:, :, 2].max(0)
        with np.errstate(invalid="ignore"):
            s_t = (s[:, :, 1] * np.exp(s[:, :, 0] - m_t)).sum(0)
            s_d = (s[:, :, 3] * np.exp(s[:, :, 2] - m_d)).sum(0)
        return (torch.from_numpy(np.stack([m_t, s_t, m_d, s_d], 1)),
                torch.from_numpy(tok_all.numpy().max(0)))

    def race(target, draft, v_off, V_total, target_row0, draft_row0, draft_len, gmax, toks, seed,
             stats, tok, request_ids=None):
        st, tk = stats.numpy(), tok.numpy()
        acc = np.zeros(B, np.int32)
        win = np.full((B, 2), -np.inf)
        for r in range(B):
            g = int(lay["draft_len"][r])
            tau = g
            for i in range(1, g + 1):
                u = r * gmax + i - 1
                p = math.exp(tk[u, 0] - st[u, 0]) / st[u, 1]
                q = math.exp(tk[u, 1] - st[u, 2]) / st[u, 3]
                if not orc.uniform(seed, r, i, orc.TAG_ACCEPT, 0) < p / q:
                    tau = i - 1
                    break
            acc[r] = tau
            row = int(lay["target_row0"][r]) + tau
            if tau < g:
                drow = draft[int(lay["draft_row0"][r]) + tau]
                key, idx = orc.race_shard(target[row], drow, v_off, 1, 1.0,
                                          st[r * gmax + tau], seed, r, tau + 1, orc.TAG_RESID)
            else:
                _, M, S = orc.row_stats(t_rows[row])  # the bonus row, unsharded statistics
                key, idx = orc.race_shard(target[row], None, v_off, 0, 1.0, (M, S, 0, 1), seed,
                                          r, tau + 1, orc.TAG_BONUS)
            win[r] = (key, idx)
        return {"accepted_len": torch.from_numpy(acc), "winners": torch.from_numpy(win)}

    def finish(winners_all, accepted_len, draft_row0, toks, out_ld):
        w = winners_all.numpy()
        out = np.full((B, out_ld), -1, np.int32)
        for r in range(B):
            keys, idxs = w[:, r, 0], w[:, r, 1]
            best = max(range(len(keys)), key=lambda k: (keys[k], -idxs[k]))
            tau = int(accepted_len[r])
            out[r, :tau] = toks[int(lay["draft_row0"][r]): int(lay["draft_row0"][r]) + tau]
            out[r, tau] = int(idxs[best])
        return {"out_tokens": torch.from_numpy(out), "accepted_len": accepted_len}

    return {"stats": stats, "merge": merge, "race": race, "finish": finish}


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    import speculative_decoding_verification_token_gb300 as sv
    w, inp = _inputs()
    lay = {k: inp[k].numpy() for k in ("target_row0", "draft_row0", "draft_len")}
    t_rows, d_rows = inp["target"].numpy(), inp["draft"].numpy()
    st, tokens = oracle.sample_draft_batch(d_rows, V, V, lay["draft_row0"], lay["draft_len"], B,
                                           SEED)
    lo, hi = (0, SPLIT) if rank == 0 else (SPLIT, V)
    got = sv.spec_verify_token_sharded(
        np.ascontiguousarray(t_rows[:, lo:hi]), np.ascontiguousarray(d_rows[:, lo:hi]), lo, V,
        lay["target_row0"], lay["draft_row0"], lay["draft_len"], G, tokens, SEED,
        steps=_oracle_steps(oracle, t_rows, d_rows, lay, tokens))
    ref = oracle.verify_batch(0, t_rows, d_rows, V, V, lay["target_row0"], lay["draft_row0"],
                              lay["draft_len"], tokens, B, SEED, out_ld=G + 1)
    out[rank] = (got["accepted_len"].numpy().tolist(), got["out_tokens"].numpy().tolist(),
                 ref["accepted_len"].tolist(), ref["out_tokens"].tolist(),
                 ref["decision_margin"].tolist(), ref["race_margin"].tolist())
    dist.barrier()
    dist.destroy_process_group()


def test_two_shards_over_gloo_match_unsharded_oracle():
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    assert res[0][:2] == res[1][:2]  # every rank ends with the same outputs
    acc, toks, racc, rtoks, dmar, rmar = (np.array(v) for v in res[0])
    exempt = (dmar < 1e-9) | (rmar < 1e-9)
    same = (acc == racc) & (toks == rtoks).all(axis=1)
    assert (same | exempt).all() and same.sum() >= B - 1, (acc, racc)
    assert (acc < np.array([4] * B)).any()  # residual races were exercised
