"""spec_verify_token_noalloc: token-level verification for callers that cannot allocate device
memory (for example a plugin that its host engine hands only input and output buffers, or a serving
loop where cudaMalloc could synchronise the device).  Called through the C ABI, its results must
equal spec_verify_token's on the same inputs, on two calls in a row (the second call reuses the
library's scratch array left behind by the first)."""
import ctypes as C

import numpy as np
import pytest
import torch

from parity import oracle_tokens
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


def _call_noalloc(sv, d, tokens, acc, out, corr, ratio, status, B=None, V=None, gmax=None):
    stream = torch.cuda.current_stream().cuda_stream
    return sv.lib().spec_verify_token_noalloc(
        d["target"].data_ptr(), d["draft"].data_ptr(), sv.SV_BF16, V or d["V"],
        d["target"].stride(0), d["target_row0"].data_ptr(), d["draft_row0"].data_ptr(),
        d["draft_len"].data_ptr(), gmax or d["max_draft_len"], tokens.data_ptr(),
        B if B is not None else d["B"], d["seed"], None, acc.data_ptr(), out.data_ptr(),
        out.shape[1], corr.data_ptr(), ratio.data_ptr(), status.data_ptr(), stream)


def test_noalloc_matches_workspace_version(sv, orc):
    w = synth.scaled(synth.TOKEN_LARGE, B=24, V=60000)
    inp = synth.token_inputs(w, device="cpu")
    tokens = torch.from_numpy(oracle_tokens(orc, inp)).cuda()
    d = dict(inp)
    for k in ("target", "draft", "target_row0", "draft_row0", "draft_len"):
        d[k] = inp[k].cuda()
    ref = sv.spec_verify_token(d["target"], d["draft"], d["target_row0"], d["draft_row0"],
                               d["draft_len"], w.gamma, tokens, w.seed)
    torch.cuda.synchronize()
    assert int(ref["status"].item()) == 0
    for call in range(2):
        acc = torch.full((w.B,), -7, dtype=torch.int32, device="cuda")
        out = torch.full((w.B, w.gamma + 1), -7, dtype=torch.int32, device="cuda")
        corr = torch.full((w.B,), -7, dtype=torch.int32, device="cuda")
        ratio = torch.full((tokens.numel(),), -7.0, device="cuda")
        status = torch.full((1,), 99, dtype=torch.int32, device="cuda")
        code = _call_noalloc(sv, d, tokens, acc, out, corr, ratio, status)
        assert code == sv.SV_OK, sv.status_string(code)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(acc, ref["accepted_len"])
        assert torch.equal(out, ref["out_tokens"])
        assert torch.equal(corr, ref["correction"])
        # same kernels on the same data: the ratios agree well inside the 1e-5 parity tolerance
        rel = (ratio - ref["accept_ratio"]).abs() / ref["accept_ratio"].abs().clamp_min(1e-6)
        assert float(rel.max()) < 1e-5


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
