"""GPU parity of dspark_markov_draft with the CPU oracle (DSpark Markov-head drafting).

Both sides get the same seeded synthetic backbone logits, factors U, W and anchors (synth).  The
oracle runs free (its own samples feed its next position), so a request is compared position by
position up to its first differing token; that token must be a near tie of the oracle's race
(a one-ulp difference of a bf16 logit can decide only a race whose top two keys lie within a few
ulps), such divergences are counted and bounded, and the request's later positions are skipped.
Compared per position: every z entry within one bf16 ulp plus the fp32 accumulation bound of the
GEMM (below; mismatches counted), the token exactly, max z within that bound, log-sum-exp within
1e-5 relative, the confidence within 1e-6.

z tolerance.  The oracle rounds the exact sum backbone + sum_j U_j W_jv once to bf16; the kernel
accumulates the 256 bf16 products in fp32 (tensor cores), adds the backbone in fp32 and rounds.
Recursive fp32 summation of n terms errs by at most n * 2^-24 * sum |terms| (first order), so the
pre-rounding values differ by at most (R + 1) * 2^-24 * (sum_j |U_j W_jv| + |backbone_v|), and the
two roundings add at most one ulp of the result.  Near z = 0 that bound spans several bf16 ulps.

Log-sum-exp tolerance.  A one-ulp difference of a heavily weighted z entry moves the log-sum-exp by
far more than the arithmetic of the statistics does, so the z differences are carried through: by
the mean value theorem |lse(z_gpu) - lse(z_oracle)| <= sum_v p_t(v) |dz_v| with p_t the softmax at
an intermediate point, and p_t(v) <= p_oracle(v) * exp(2 max |dz|).  The test allows that plus
1e-5 relative for the kernel's own fp32 statistics."""
import numpy as np
import pytest
import torch

from speculative_decoding_verification_token_gb300 import synth

pytestmark = pytest.mark.gpu

LSE_REL = 1e-5
CONF_ABS = 1e-6


@pytest.fixture(scope="module")
def sv():
    import speculative_decoding_verification_token_gb300 as sv
    from speculative_decoding_verification_token_gb300 import build
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    return sv


def _bf16_bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().astype(np.uint16)


def _ulp(x):
    x = max(abs(float(x)), 1e-30)
    return 2.0 ** (np.floor(np.log2(x)) - 7)


def run_markov(sv, inp, request_ids=None, **kw):
    out = sv.dspark_markov_draft(inp["backbone"], inp["U"], inp["Wt"], inp["anchor"],
                                 inp["scores"], inp["T"], inp["seed"], request_ids=request_ids,
                                 **kw)
    torch.cuda.synchronize()
    return out


def _bf16_values(bits):
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()


def _ulps(x):
    """One bf16 ulp of |x| (elementwise; subnormal floor 2^-133)."""
    e = np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** -126)))
    return 2.0 ** (e - 7)


def compare_markov(orc, inp_cpu, out, reqs, request_ids=None, workers=1):
    """Compares the GPU draft of the requests `reqs` with the oracle; returns counters.  The
    oracle runs on `workers` host threads (its C calls release the interpreter lock)."""
    import concurrent.futures as cf
    U = inp_cpu["U"].float().numpy()
    W = inp_cpu["W"].float().numpy()
    absW = np.abs(W.astype(np.float64))
    R = U.shape[1]
    T = inp_cpu["T"].numpy()
    x_gpu = out["draft_tokens"].cpu().numpy()
    z_gpu = out["draft_logits"]
    stats = out["row_stats"].cpu().numpy()
    conf = out["conf"].cpu().numpy() if out["conf"] is not None else None
    K = x_gpu.shape[1]
    n = {"rows": 0, "z_entries": 0, "z_mismatch": 0, "divergent": 0}

    def oracle_of(b):
        req = int(request_ids[b]) if request_ids is not None else int(b)
        return orc.markov_draft_request(inp_cpu["backbone"][b].float().numpy(), U, W,
                                        int(inp_cpu["anchor"][b]), inp_cpu["scores"][b].numpy(),
                                        T, inp_cpu["seed"], req)
    reqs = list(reqs)
    with cf.ThreadPoolExecutor(max_workers=max(1, workers)) as ex:
        refs = list(ex.map(oracle_of, reqs))
    for b, o in zip(reqs, refs):
        assert o["status"] == 0
        zb = _bf16_bits(z_gpu[b])
        bb = inp_cpu["backbone"][b].double().numpy()
        for k in range(K):
            prev = int(inp_cpu["anchor"][b]) if k == 0 else int(o["x"][k - 1])
            acc_err = (R + 1) * 2.0 ** -24 * (np.abs(U[prev].astype(np.float64)) @ absW
                                             + np.abs(bb[k]))
            zg, zo = _bf16_values(zb[k]), _bf16_values(o["z"][k])
            tol = _ulps(np.maximum(np.abs(zg), np.abs(zo))) + acc_err
            bad = np.abs(zg - zo) > tol
            assert not bad.any(), (b, k, np.flatnonzero(bad)[:5], zg[bad][:5], zo[bad][:5])
            n["z_mismatch"] += int((zb[k] != o["z"][k]).sum())
            n["z_entries"] += zb[k].size
            n["rows"] += 1
            zmax, lse = o["stats"][k]
            assert abs(stats[b, k, 0] - zmax) <= _ulp(zmax) + acc_err.max(), (b, k)
            dz = np.abs(zg - zo)
            carried = np.exp(2 * dz.max()) * float(np.exp(zo - lse) @ dz)
            assert abs(stats[b, k, 1] - lse) <= LSE_REL * max(1.0, abs(lse)) + carried, (b, k)
            if conf is not None:
                assert abs(conf[b, k] - o["conf"][k]) <= CONF_ABS, (b, k)
            if x_gpu[b, k] != o["x"][k]:
                tol = 2 * _ulp(zmax) + 1e-4
                assert o["margin"][k] < tol, (b, k, int(x_gpu[b, k]), int(o["x"][k]),
                                              o["margin"][k])
                n["divergent"] += 1
                break
    return n


def _device(inp):
    d = dict(inp)
    for k in ("backbone", "U", "W", "Wt", "anchor", "scores", "T"):
        d[k] = inp[k].cuda()
    return d


def test_markov_small_parity(sv, orc):
    """200 requests (two M-blocks, the second ragged) x 3 positions x V = 1000 (ragged tile)."""
    inp = synth.markov_inputs(synth.MARKOV_SMALL)
    out = run_markov(sv, _device(inp))
    assert int(out["status"].item()) == 0
    n = compare_markov(orc, inp, out, range(inp["B"]))
    assert n["divergent"] <= 2, n
    assert n["z_mismatch"] <= 1e-3 * n["z_entries"], n


def test_markov_request_ids_and_padding(sv, orc):
    """uint64 request ids with high bits, backbone rows padded to ldb > V (V % 8 != 0) and Wt rows
    padded to ldw > R."""
    w = synth.MarkovWorkload("markov_pad", 131, 4, 1001, 256, 2.0, 0.25, 11, 1007)
    inp = synth.markov_inputs(w)
    ldb, ldw = 1008, 264
    bb = torch.zeros((w.B, w.K, ldb), dtype=torch.bfloat16)
    bb[:, :, : w.V] = inp["backbone"]
    wt = torch.zeros((w.V, ldw), dtype=torch.bfloat16)
    wt[:, : w.R] = inp["Wt"]
    dev = _device(inp)
    dev["backbone"] = bb.cuda()[:, :, : w.V]
    dev["Wt"] = wt.cuda()[:, : w.R]
    rng = np.random.default_rng(5)
    ids = rng.integers(0, 2**63, size=w.B, dtype=np.uint64) | np.uint64(1 << 62)
    out = run_markov(sv, dev, request_ids=torch.from_numpy(ids.view(np.int64)).cuda())
    assert int(out["status"].item()) == 0
    n = compare_markov(orc, inp, out, range(w.B), request_ids=ids)
    assert n["divergent"] <= 2, n


def test_markov_optional_outputs_and_determinism(sv):
    inp = _device(synth.markov_inputs(synth.MARKOV_SMALL))
    a = run_markov(sv, inp)
    b = run_markov(sv, inp)
    assert torch.equal(a["draft_tokens"], b["draft_tokens"])
    assert torch.equal(a["draft_logits"].view(torch.int16), b["draft_logits"].view(torch.int16))
    assert torch.equal(a["row_stats"], b["row_stats"])
    c = sv.dspark_markov_draft(inp["backbone"], inp["U"], inp["Wt"], inp["anchor"], None, None,
                               inp["seed"], want_logits=False, want_stats=False)
    torch.cuda.synchronize()
    assert int(c["status"].item()) == 0
    assert torch.equal(a["draft_tokens"], c["draft_tokens"])


def test_markov_bad_anchor_reports(sv):
    inp = _device(synth.markov_inputs(synth.MARKOV_SMALL))
    inp["anchor"][7] = inp["V"]  # one past the vocabulary
    out = run_markov(sv, inp)
    assert int(out["status"].item()) == sv.SV_ERR_BAD_INPUT
    toks = out["draft_tokens"]
    assert bool(((toks >= 0) & (toks < inp["V"])).all())


def test_markov_rejects_unsupported(sv):
    inp = _device(synth.markov_inputs(synth.MARKOV_SMALL))
    with pytest.raises(sv.SpecVerifyError) as e:
        sv.dspark_markov_draft(inp["backbone"], inp["U"][:, :128].contiguous(),
                               inp["Wt"][:, :128].contiguous(), inp["anchor"], inp["scores"],
                               inp["T"], inp["seed"])
    assert e.value.code == sv.SV_ERR_UNSUPPORTED


def test_markov_full_size_sampled(sv, orc):
    """256 requests x 16 positions x V = 151936, R = 256, in the configuration the benchmark
    times; the oracle checks 32 requests spread over both 128-request M-blocks (the first and
    last row of each among them), every request is checked through properties of its own
    outputs."""
    import os
    w = synth.MARKOV
    inp = synth.markov_inputs(w, device="cuda")
    out = run_markov(sv, inp)
    assert int(out["status"].item()) == 0
    x = out["draft_tokens"]
    assert bool(((x >= 0) & (x < w.V)).all())
    # properties at every row: the statistics describe the returned logits
    z = out["draft_logits"].float()
    assert torch.equal(out["row_stats"][..., 0], z.amax(dim=-1))
    lse = torch.logsumexp(z.double(), dim=-1)
    rel = ((out["row_stats"][..., 1].double() - lse).abs() / lse.abs().clamp(min=1.0)).max()
    assert float(rel) <= LSE_REL
    del z, lse
    half = list(range(0, 127, 9)) + [127]   # 16 requests of the first M-block, ends included
    reqs = half + [128 + b for b in half]
    cpu = {"backbone": inp["backbone"][reqs].cpu(), "U": inp["U"].cpu(), "W": inp["W"].cpu(),
           "anchor": inp["anchor"][reqs].cpu(), "scores": inp["scores"][reqs].cpu(),
           "T": inp["T"].cpu(), "seed": inp["seed"]}
    sub = {"draft_tokens": x[reqs], "draft_logits": out["draft_logits"][reqs],
           "row_stats": out["row_stats"][reqs], "conf": out["conf"][reqs]}
    ids = np.array(reqs, dtype=np.uint64)
    n = compare_markov(orc, cpu, sub, range(len(reqs)), request_ids=ids,
                       workers=os.cpu_count() or 1)
    print(f"\n[parity] markov full size, {len(reqs)} requests: {n}")
    assert len(reqs) == 32 and min(reqs) < 128 <= max(reqs)
    assert n["divergent"] <= 2, n
    assert n["rows"] >= 28 * w.K, n
