"""Failure detection on the GPU without a fault: the bounded waits every kernel uses are made to
run out (a barrier phase nobody completes, a word nobody publishes), report SV_ERR_TIMEOUT through
the status word, and leave the context usable for the next call."""
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


@pytest.mark.parametrize("which", [0, 1])
def test_bounded_wait_times_out(sv, which):
    status = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    sv.sv_selftest_wait(which, 20000, status)  # 20 ms instead of the kernels' one second
    stop.record()
    torch.cuda.synchronize()
    assert int(status.item()) == sv.SV_ERR_TIMEOUT
    assert 15.0 <= start.elapsed_time(stop) < 1000.0


def test_context_usable_after_timeouts(sv, orc):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sv.sv_selftest_wait(0, 5000, status)
    sv.sv_selftest_wait(1, 5000, status)
    torch.cuda.synchronize()
    inp = synth.token_inputs(synth.TOKEN_SMALL, device="cpu")
    tokens = oracle_tokens(orc, inp)
    ref = oracle_verify(orc, 0, inp, tokens)
    d = {k: inp[k].cuda() for k in ("target", "draft", "target_row0", "draft_row0", "draft_len")}
    out = sv.spec_verify_token(d["target"], d["draft"], d["target_row0"], d["draft_row0"],
                               d["draft_len"], inp["max_draft_len"], torch.from_numpy(tokens).cuda(),
                               inp["seed"])
    torch.cuda.synchronize()
    assert int(out["status"].item()) == 0
    lay = layout_np(inp)
    compare_verify(out, ref, 0, lay["draft_len"], lay["draft_row0"])


def test_selftest_argument_errors(sv):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for which, limit in ((2, 1000), (0, 0), (1, 2000000)):
        with pytest.raises(sv.SpecVerifyError):
            sv.sv_selftest_wait(which, limit, status)
