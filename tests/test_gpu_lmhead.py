"""GPU parity of spec_verify_lmhead (verification from hidden states) with the CPU oracle.

Both sides get the same seeded hidden rows and output projection (synth.lmhead_inputs) and the
same drafted tokens, sampled from q by the oracle.  The oracle's logits are binary64 sums rounded
once to binary32 (oracle.lmhead_logits); the GPU's are the tensor cores' fp32 sums of the same
bf16 products, so the two sides' logits differ by rounding and the comparison widens the
near-tie margins and the ratio tolerance accordingly (LOGIT_TIE, RATIO_TOL)."""
import numpy as np
import pytest
import torch

from parity import compare_verify
from speculative_decoding_verification_token_gb300 import synth

pytestmark = pytest.mark.gpu

# A logit is a sum of H products; the two sides add them in different orders and precisions.
# With H <= 2560 products of magnitude |h||w| <~ 0.3, fp32 accumulation moves a logit by a few
# 1e-5, and p(x)/q(x) = exp(t_x - d_x) Z_d / Z_t inherits at most four such errors.  Decisions
# and races whose oracle margin is below LOGIT_TIE are exempt (counted, at most 1% may differ).
LOGIT_TIE = 1e-3
RATIO_TOL = 1e-3


@pytest.fixture(scope="module")
def sv():
    import speculative_decoding_verification_token_gb300 as sv
    from speculative_decoding_verification_token_gb300 import build
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    return sv


def _oracle_logits(orc, inp):
    tl = orc.lmhead_logits(inp["target_hidden"].float().numpy(), inp["W"].float().numpy())
    dl = orc.lmhead_logits(inp["draft_hidden"].float().numpy(), inp["W"].float().numpy())
    return tl, dl


def _oracle_drafts(orc, inp, dl):
    st, toks = orc.sample_draft_batch(dl, inp["V"], dl.shape[1], inp["draft_row0"].numpy(),
                                      inp["draft_len"].numpy(), inp["B"], inp["seed"])
    assert st == 0
    return toks


def _gpu(sv, inp, tokens, request_ids=None):
    d = {k: inp[k].cuda() for k in ("target_hidden", "draft_hidden", "W", "target_row0",
                                     "draft_row0", "draft_len")}
    out = sv.spec_verify_lmhead(d["target_hidden"], d["draft_hidden"], d["W"], d["target_row0"],
                                d["draft_row0"], d["draft_len"], inp["max_draft_len"],
                                torch.from_numpy(tokens).cuda(), inp["seed"],
                                request_ids=request_ids)
    torch.cuda.synchronize()
    assert int(out["status"].item()) == 0, sv.status_string(int(out["status"].item()))
    return out


def _parity(sv, orc, inp, request_ids=None):
    tl, dl = _oracle_logits(orc, inp)
    tokens = _oracle_drafts(orc, inp, dl)
    rid = None if request_ids is None else request_ids.cpu().numpy()
    ref = orc.verify_batch(0, tl, dl, inp["V"], tl.shape[1], inp["target_row0"].numpy(),
                           inp["draft_row0"].numpy(), inp["draft_len"].numpy(), tokens,
                           inp["B"], inp["seed"], request_ids=rid,
                           out_ld=inp["max_draft_len"] + 1)
    assert ref["status"] == 0
    gpu = _gpu(sv, inp, tokens, request_ids)
    res = compare_verify(gpu, ref, False, inp["draft_len"].numpy(), inp["draft_row0"].numpy(),
                         near_tie=LOGIT_TIE, rel_tol=RATIO_TOL)
    res["recomputed"] = int(gpu["recomputed"].item())
    print(f"\n[lmhead parity] B={inp['B']} V={inp['V']} H={inp['H']}: {res}")
    return gpu, ref, res


def test_lmhead_parity_small(sv, orc):
    """Three slot blocks, 17 vocabulary tiles with a ragged last one, five k-blocks."""
    inp = synth.lmhead_inputs(synth.LMHEAD_SMALL)
    gpu, ref, res = _parity(sv, orc, inp)
    # the batch exercises both outcomes: corrections after a rejection and bonus tokens
    acc = ref["accepted_len"]
    assert (acc < inp["max_draft_len"]).any() and (acc == inp["max_draft_len"]).any()


def test_lmhead_parity_ragged_ids(sv, orc):
    """Ragged draft lengths (0 .. gamma), rows of each request placed out of order, and caller
    request ids keying the Philox streams."""
    w = synth.LmHeadWorkload("lmhead_ragged", 40, 6, 2053, 256, 3.0, 1.1, 1.0, 11, 1009)
    lens = synth.ragged_lengths(w.B, w.gamma, 77)
    inp = synth.lmhead_inputs(w, draft_len=lens)
    perm = torch.from_numpy(np.random.default_rng(4).permutation(w.B))
    inp["target_row0"] = inp["target_row0"][perm].contiguous()
    inp["draft_row0"] = inp["draft_row0"][perm].contiguous()
    rids = torch.from_numpy(np.random.default_rng(5).integers(0, 2**60, w.B).astype(np.uint64)
                            .view(np.int64)).cuda()
    _parity(sv, orc, inp, request_ids=rids)


@pytest.mark.parametrize("B,gamma,V,H", [(20, 16, 1500, 64), (7, 2, 200, 192), (33, 3, 777, 128)])
def test_lmhead_parity_shapes(sv, orc, B, gamma, V, H):
    """Requests that straddle slot blocks (34 slots per request), one k-block (H = 64), a vocabulary
    smaller than one tile (V = 200), and an odd vocabulary with odd request counts."""
    w = synth.LmHeadWorkload("lmhead_shape", B, gamma, V, H, 3.0, 1.1, 1.0, 14 + B, 1013 + B)
    _parity(sv, orc, synth.lmhead_inputs(w))


def test_lmhead_no_drafts(sv, orc):
    """max_draft_len = 0: every request takes its bonus token from target row 0."""
    w = synth.LmHeadWorkload("lmhead_nodraft", 9, 0, 1500, 128, 3.0, 1.1, 1.0, 12, 1010)
    inp = synth.lmhead_inputs(w)
    gpu, ref, _ = _parity(sv, orc, inp)
    assert (gpu["accepted_len"].cpu().numpy() == 0).all()


def _adversarial_inputs(B, gamma, V, H, seed, gen_seed):
    """Hidden rows whose residual mass hides behind the largest plain keys.  Logits are N(0, 1)
    except the 32 tokens {0..15, 32..47}: target logit 7 (+ N(0, 0.3^2)), draft logit 4 higher.
    The draft puts almost all of q on those tokens, so a drafted token is rejected with
    probability about 0.08 per position, and the correction then comes from the other tokens,
    whose plain keys sit far below the top tokens' -- the case the first pass's candidates often
    cannot settle, so the correction is recomputed.  Column 0 carries the constant logit offsets,
    column 1 the draft's extra offset, the rest the N(0, 1) part."""
    g = torch.Generator().manual_seed(gen_seed)
    top = torch.zeros(V, dtype=torch.bool)
    top[0:16] = True
    top[32:48] = True
    W = torch.randn((V, H), generator=g) / np.sqrt(H - 2)
    W[:, 0] = 0.0
    W[:, 1] = 0.0
    W[top, 0] = 7.0
    W[top, 1] = 4.0
    W[top, 2:] *= 0.3
    target = torch.randn((B * (gamma + 1), H), generator=g)
    target[:, 0] = 1.0
    target[:, 1] = 0.0
    draft = target.view(B, gamma + 1, H)[:, :gamma, :].reshape(B * gamma, H).clone()
    draft[:, 1] = 1.0
    return {
        "target_hidden": target.to(torch.bfloat16), "draft_hidden": draft.to(torch.bfloat16),
        "W": W.to(torch.bfloat16), "V": V, "H": H,
        "target_row0": torch.arange(B, dtype=torch.int64) * (gamma + 1),
        "draft_row0": torch.arange(B, dtype=torch.int64) * gamma,
        "draft_len": torch.full((B,), gamma, dtype=torch.int32),
        "max_draft_len": gamma, "B": B, "seed": seed,
    }


def test_lmhead_recomputed_corrections(sv, orc):
    """Corrections the candidates cannot settle go through the second pass, and agree with the
    oracle like the rest."""
    inp = _adversarial_inputs(48, 6, 2053, 192, 21, 1011)
    gpu, ref, res = _parity(sv, orc, inp)
    n = int(gpu["recomputed"].item())
    print(f"[lmhead] recomputed corrections: {n} of {inp['B']}")
    assert n > 0
    assert n <= int((ref["accepted_len"] < inp["max_draft_len"]).sum())


def test_lmhead_full_size_sampled(sv, orc):
    """64 requests x 5 positions, V = 151936, H = 2560, in the launch configuration the benchmark
    times; two requests checked against the oracle, every request against the invariants."""
    w = synth.LMHEAD
    inp = {k: (v.cpu() if torch.is_tensor(v) else v)
           for k, v in synth.lmhead_inputs(w, device="cuda").items()}
    B, G, V = w.B, w.gamma, w.V
    Wf = inp["W"].float().numpy()
    picks = [3, 41]
    # drafted tokens: the oracle's sampler for the checked requests, torch's for the others
    dh = inp["draft_hidden"].cuda().float()
    dlog = dh @ inp["W"].cuda().float().t()
    tokens = torch.multinomial(torch.softmax(dlog, dim=1), 1,
                               generator=torch.Generator(device="cuda").manual_seed(5))
    tokens = tokens.view(-1).to(torch.int32).cpu().numpy()
    del dlog, dh
    sub = {}
    for r in picks:
        th = inp["target_hidden"][r * (G + 1):(r + 1) * (G + 1)].float().numpy()
        dhr = inp["draft_hidden"][r * G:(r + 1) * G].float().numpy()
        tl = orc.lmhead_logits(th, Wf)
        dl = orc.lmhead_logits(dhr, Wf)
        for i in range(G):
            _, tok, _ = orc.sample_race(dl[i], w.seed, r, i + 1, orc.TAG_DRAFT)
            tokens[r * G + i] = tok
        sub[r] = (tl, dl)
    gpu = _gpu(sv, inp, tokens)
    acc = gpu["accepted_len"].cpu().numpy()
    out = gpu["out_tokens"].cpu().numpy()
    assert ((acc >= 0) & (acc <= G)).all()
    for r in range(B):
        assert (out[r, :acc[r]] == tokens[r * G:r * G + acc[r]]).all()
        assert 0 <= out[r, acc[r]] < V
        assert (out[r, acc[r] + 1:] == -1).all()
    for r in picks:
        tl, dl = sub[r]
        ref = orc.verify_batch(0, tl, dl, V, V, np.array([0]), np.array([0]),
                               np.array([G], np.int32), tokens[r * G:(r + 1) * G], 1, w.seed,
                               request_ids=np.array([r], np.uint64), out_ld=G + 1)
        assert ref["status"] == 0
        tie = ref["decision_margin"][0] < LOGIT_TIE or ref["race_margin"][0] < LOGIT_TIE
        same = acc[r] == ref["accepted_len"][0] and (out[r] == ref["out_tokens"][0]).all()
        assert same or tie, (r, acc[r], ref["accepted_len"][0], out[r], ref["out_tokens"][0])
        ratio = gpu["accept_ratio"].cpu().numpy()[r * G:(r + 1) * G]
        rel = np.abs(ratio - ref["ratio"]) / np.maximum(np.abs(ref["ratio"]), 1e-6)
        assert np.all(rel < RATIO_TOL), rel


def test_lmhead_rejects_bad_shapes(sv):
    """H not a multiple of 64 is refused before any launch."""
    dev = "cuda"
    th = torch.zeros((2, 96), dtype=torch.bfloat16, device=dev)
    W = torch.zeros((100, 96), dtype=torch.bfloat16, device=dev)
    z = torch.zeros(1, dtype=torch.int64, device=dev)
    with pytest.raises(sv.SpecVerifyError):
        sv.spec_verify_lmhead(th, th, W, z, z, torch.zeros(1, dtype=torch.int32, device=dev), 0,
                              torch.zeros(1, dtype=torch.int32, device=dev), 0)
