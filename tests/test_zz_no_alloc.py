"""spec_verify_token_noalloc: token-level verification for callers that cannot allocate device
memory (for example a plugin that its host engine hands only input and output buffers, or a serving
loop where cudaMalloc could synchronise the device).  Called through the C ABI, its results must
equal spec_verify_token's on the same inputs, and the oracle's, on two calls in a row (the second
call reuses the library's scratch array left behind by the first): on a small ragged batch, with
no drafted tokens at all, at the 64 x 5 x 151936 benchmark size, and at the largest batch whose
scratch fits the array, whose neighbour one request larger is refused."""
import ctypes as C

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


def _call_noalloc(sv, d, tokens, acc, out, corr, ratio, status, B=None, V=None, gmax=None,
                  dtype=None):
    stream = torch.cuda.current_stream().cuda_stream
    if dtype is None:
        dtype = sv.SV_BF16 if d["target"].dtype == torch.bfloat16 else sv.SV_F32
    return sv.lib().spec_verify_token_noalloc(
        d["target"].data_ptr(), d["draft"].data_ptr(), dtype, V or d["V"],
        d["target"].stride(0), d["target_row0"].data_ptr(), d["draft_row0"].data_ptr(),
        d["draft_len"].data_ptr(), gmax or d["max_draft_len"], tokens.data_ptr(),
        B if B is not None else d["B"], d["seed"], None, acc.data_ptr(), out.data_ptr(),
        out.shape[1], corr.data_ptr(), ratio.data_ptr(), status.data_ptr(), stream)


def _device(inp):
    d = dict(inp)
    for k in ("target", "draft", "target_row0", "draft_row0", "draft_len"):
        d[k] = inp[k].cuda()
    return d


def _check_twice(sv, orc, inp, tokens_np, dtype=None):
    """Two allocation-free calls in a row, each equal to spec_verify_token and to the oracle."""
    d = _device(inp)
    B, G = inp["B"], inp["max_draft_len"]
    tokens = torch.from_numpy(tokens_np).cuda()
    ref = sv.spec_verify_token(d["target"], d["draft"], d["target_row0"], d["draft_row0"],
                               d["draft_len"], G, tokens, inp["seed"])
    torch.cuda.synchronize()
    assert int(ref["status"].item()) == 0
    orc_ref = oracle_verify(orc, 0, inp, tokens_np)
    assert orc_ref["status"] == 0
    lay = layout_np(inp)
    for call in range(2):
        acc = torch.full((B,), -7, dtype=torch.int32, device="cuda")
        out = torch.full((B, G + 1), -7, dtype=torch.int32, device="cuda")
        corr = torch.full((B,), -7, dtype=torch.int32, device="cuda")
        ratio = torch.full((max(1, tokens.numel()),), -7.0, device="cuda")
        status = torch.full((1,), 99, dtype=torch.int32, device="cuda")
        code = _call_noalloc(sv, d, tokens, acc, out, corr, ratio, status, dtype=dtype)
        assert code == sv.SV_OK, sv.status_string(code)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(acc, ref["accepted_len"])
        assert torch.equal(out, ref["out_tokens"])
        assert torch.equal(corr, ref["correction"])
        if G > 0:
            # same kernels on the same data: the ratios of every drafted row agree well inside
            # the 1e-5 tolerance (rows past a request's drafted length are not written)
            rows = torch.from_numpy(np.concatenate(
                [np.arange(r0, r0 + g) for r0, g in zip(lay["draft_row0"], lay["draft_len"])]
                + [np.zeros(0, np.int64)]).astype(np.int64)).cuda()
            a, b = ratio[rows], ref["accept_ratio"][rows]
            rel = (a - b).abs() / b.abs().clamp_min(1e-6)
            assert rows.numel() == 0 or float(rel.max()) < 1e-5
        got = {"accepted_len": acc, "out_tokens": out,
               "accept_ratio": ratio if G > 0 else None}
        compare_verify(got, orc_ref, 0, lay["draft_len"], lay["draft_row0"])


def test_noalloc_matches_workspace_version(sv, orc):
    w = synth.scaled(synth.TOKEN_LARGE, B=24, V=60000)
    inp = synth.token_inputs(w, device="cpu", draft_len=synth.ragged_lengths(24, w.gamma, 2))
    _check_twice(sv, orc, inp, oracle_tokens(orc, inp))


def test_noalloc_without_drafts(sv, orc):
    """max_draft_len = 0: every request takes only its bonus token."""
    w = synth.scaled(synth.TOKEN_LARGE, B=6, gamma=0, V=9000)
    inp = synth.token_inputs(w, device="cpu")
    _check_twice(sv, orc, inp, np.zeros(1, np.int32))


def test_noalloc_benchmark_size(sv, orc):
    """The 64 x 5 x 151936 bf16 benchmark workload fits the array."""
    w = synth.TOKEN_LARGE
    assert sv.spec_verify_workspace_bytes(w.B, w.gamma, w.V, sv.SV_BF16) <= sv.SV_NOALLOC_SCRATCH_BYTES
    inp = synth.token_inputs(w, device="cpu")
    _check_twice(sv, orc, inp, oracle_tokens(orc, inp))


def test_noalloc_largest_batch_that_fits(sv, orc):
    """With 64 drafted positions of V = 64 bf16 per request the scratch grows with the batch: the
    largest batch whose spec_verify_workspace_bytes fits the array runs and matches, the batch one
    request larger is refused with SV_ERR_UNSUPPORTED before anything launches."""
    G, V = 64, 64
    cap = sv.SV_NOALLOC_SCRATCH_BYTES

    def need(b):
        return sv.spec_verify_workspace_bytes(b, G, V, sv.SV_BF16)
    lo, hi = 1, 1
    while need(hi) <= cap:
        lo, hi = hi, hi * 2
    while hi - lo > 1:
        mid = (lo + hi) // 2
        lo, hi = (mid, hi) if need(mid) <= cap else (lo, mid)
    B = lo
    assert need(B) <= cap < need(B + 1)
    w = synth.scaled(synth.TOKEN_LARGE, B=B + 1, gamma=G, V=V, draft_noise=0.3)
    inp = synth.token_inputs(w, device="cpu")
    d = _device(inp)
    t = torch.zeros(max(1, (B + 1) * G), dtype=torch.int32, device="cuda")
    o = torch.zeros((B + 1, G + 1), dtype=torch.int32, device="cuda")
    a = torch.zeros(B + 1, dtype=torch.int32, device="cuda")
    f = torch.zeros((B + 1) * G, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert _call_noalloc(sv, d, t, a, o, a, f, st, B=B + 1) == sv.SV_ERR_UNSUPPORTED
    inp = synth.token_inputs(synth.scaled(w, B=B), device="cpu")
    _check_twice(sv, orc, inp, oracle_tokens(orc, inp))


def test_noalloc_rejects_batches_beyond_its_scratch(sv):
    """A batch whose scratch would exceed the fixed array is refused before anything launches."""
    need = sv.spec_verify_workspace_bytes(65536, 64, 262144, sv.SV_BF16)
    assert need > (8 << 20)
    dummy = {"target": torch.zeros((1, 8), dtype=torch.bfloat16, device="cuda"),
             "draft": torch.zeros((1, 8), dtype=torch.bfloat16, device="cuda"),
             "target_row0": torch.zeros(1, dtype=torch.int64, device="cuda"),
             "draft_row0": torch.zeros(1, dtype=torch.int64, device="cuda"),
             "draft_len": torch.zeros(1, dtype=torch.int32, device="cuda"),
             "V": 8, "max_draft_len": 1, "B": 1, "seed": 0}
    t = torch.zeros(1, dtype=torch.int32, device="cuda")
    f = torch.zeros(1, device="cuda")
    o = torch.zeros((1, 65), dtype=torch.int32, device="cuda")
    code = _call_noalloc(sv, dummy, t, t, o, t, f, t, B=65536, V=262144, gmax=64)
    assert code == sv.SV_ERR_UNSUPPORTED
