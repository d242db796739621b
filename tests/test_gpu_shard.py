"""GPU parity of vocabulary-sharded token verification (spec_verify_shard_*): the rows split into
2 or 3 vocabulary shards (offsets multiples of 8), each shard's statistics and race computed by the
library's kernels, the exchanges done by stacking the shards' outputs in shard order (as an
all-gather over ranks would).  Accepted lengths and emitted tokens must equal the oracle's
verification of the unsharded rows (near ties exempt, counted) and the unsharded GPU call's."""
import numpy as np
import pytest
import torch

from parity import compare_verify, layout_np, oracle_tokens, oracle_verify
from speculative_decoding_verification_token_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    import speculative_decoding_verification_token_gb300 as sv
    from speculative_decoding_verification_token_gb300 import build
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    return sv


def _sharded(sv, inp, tokens, cuts):
    """The four shard calls over the shards [cuts[k], cuts[k + 1]) of every row."""
    d = {k: inp[k].cuda() for k in ("target_row0", "draft_row0", "draft_len")}
    tok = torch.from_numpy(tokens).cuda()
    V, G = inp["V"], inp["max_draft_len"]
    shards = []
    for lo, hi in zip(cuts[:-1], cuts[1:]):
        ld = (hi - lo + 7) // 8 * 8
        t = torch.zeros((inp["target"].shape[0], ld), dtype=inp["target"].dtype)
        dr = torch.zeros((inp["draft"].shape[0], ld), dtype=inp["draft"].dtype)
        t[:, : hi - lo] = inp["target"][:, lo:hi]
        dr[:, : hi - lo] = inp["draft"][:, lo:hi]
        shards.append((lo, t.cuda()[:, : hi - lo], dr.cuda()[:, : hi - lo]))
    parts = [sv.spec_verify_shard_stats(t, dr, lo, V, d["target_row0"], d["draft_row0"],
                                        d["draft_len"], G, tok) for lo, t, dr in shards]
    stats, tk = sv.spec_verify_shard_merge(torch.stack([p[0] for p in parts]),
                                           torch.stack([p[1] for p in parts]))
    races = [sv.spec_verify_shard_race(t, dr, lo, V, d["target_row0"], d["draft_row0"],
                                       d["draft_len"], G, tok, inp["seed"], stats, tk)
             for lo, t, dr in shards]
    for r in races[1:]:  # every shard decides the same way
        assert torch.equal(r["accepted_len"], races[0]["accepted_len"])
    out = sv.spec_verify_shard_finish(torch.stack([r["winners"] for r in races]),
                                      races[0]["accepted_len"], d["draft_row0"], tok, G + 1)
    torch.cuda.synchronize()
    for r in races:
        assert int(r["status"].item()) == 0
    assert int(out["status"].item()) == 0
    out["accept_ratio"] = races[0]["accept_ratio"]
    return out


@pytest.mark.parametrize("cuts_frac", [(0.5,), (0.27, 0.61)])
@pytest.mark.parametrize("dtype,V", [(torch.bfloat16, 40000), (torch.float32, 9000)])
def test_sharded_matches_oracle_and_unsharded(sv, orc, cuts_frac, dtype, V):
    w = synth.scaled(synth.TOKEN_LARGE, B=16, V=V, dtype=dtype)
    inp = synth.token_inputs(w, device="cpu", draft_len=synth.ragged_lengths(16, w.gamma, 5))
    tokens = oracle_tokens(orc, inp)
    cuts = [0] + [int(f * V) // 8 * 8 for f in cuts_frac] + [V]
    got = _sharded(sv, inp, tokens, cuts)
    ref = oracle_verify(orc, 0, inp, tokens)
    lay = layout_np(inp)
    res = compare_verify(got, ref, 0, lay["draft_len"], lay["draft_row0"])
    print(f"\n[parity] sharded {len(cuts) - 1} ways, V={V}: {res}")
    d = {k: inp[k].cuda() for k in ("target", "draft", "target_row0", "draft_row0", "draft_len")}
    full = sv.spec_verify_token(d["target"], d["draft"], d["target_row0"], d["draft_row0"],
                                d["draft_len"], w.gamma, torch.from_numpy(tokens).cuda(),
                                inp["seed"])
    torch.cuda.synchronize()
    assert torch.equal(full["accepted_len"], got["accepted_len"])
    assert torch.equal(full["out_tokens"], got["out_tokens"])


def test_sharded_full_size_and_empty_residual(sv, orc):
    """The 64 x 5 x 151936 bf16 workload split four ways, and requests whose correction residual
    is empty in every shard (the race over p, taken from the shards' fallback winners)."""
    w = synth.TOKEN_LARGE
    inp = synth.token_inputs(w, device="cpu")
    tokens = oracle_tokens(orc, inp)
    # requests 0 and 1: position 1 degenerate -- the target masks the drafted token, the draft
    # gives it -120, every other entry equal in both rows (p = q exactly elsewhere)
    for r in (0, 1):
        trow, drow = r * (w.gamma + 1), r * w.gamma
        x = 1000 + 70000 * r
        inp["draft"][drow] = inp["target"][trow]
        inp["target"][trow, x] = float("-inf")
        inp["draft"][drow, x] = -120.0
        tokens[drow] = x
    cuts = [0, 37984, 75968, 113952, w.V]
    got = _sharded(sv, inp, tokens, cuts)
    ref = oracle_verify(orc, 0, inp, tokens)
    assert (ref["race_kind"][:2] == orc.RACE_RESIDUAL_EMPTY).all()
    lay = layout_np(inp)
    res = compare_verify(got, ref, 0, lay["draft_len"], lay["draft_row0"])
    print(f"\n[parity] sharded 4 ways, full size: {res}")
