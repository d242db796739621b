"""The C-ABI library builds, loads, exports every function include/specverify.h declares, and
rejects invalid arguments synchronously (no GPU needed: nothing is launched)."""
import ctypes as C

import pytest


@pytest.fixture(scope="module")
def sv():
    import speculative_decoding_verification_token_gb300 as sv
    from speculative_decoding_verification_token_gb300 import build
    build.build()
    return sv


def test_exports_every_declared_symbol(sv):
    names = sv.declared_functions()
    assert {"spec_verify_token", "spec_verify_block", "dspark_markov_draft",
            "dspark_schedule"} <= set(names)
    L = sv.lib()
    for n in names:
        assert hasattr(L, n), n


def test_status_strings(sv):
    for code in range(6):
        assert sv.status_string(code).startswith("SV_")
    assert "sm_103a" in sv.version()


def test_workspace_queries(sv):
    a = sv.spec_verify_workspace_bytes(64, 5, 151936, sv.SV_BF16)
    b = sv.spec_verify_workspace_bytes(128, 7, 129280, sv.SV_BF16)
    assert 0 < a < b < 64 << 20
    assert sv.spec_verify_workspace_bytes(-1, 5, 100, sv.SV_F32) == 0
    assert sv.spec_verify_workspace_bytes(4, sv.SV_MAX_DRAFT_LEN + 1, 100, sv.SV_F32) == 0
    assert sv.dspark_schedule_workspace_bytes(512, 16) > 0


def test_invalid_arguments_rejected_before_launch(sv):
    L = sv.lib()
    fake = C.c_void_p(4096)  # never dereferenced: validation fails first
    args = dict(V=1024, ld=1024, gmax=4, B=4)

    def call(V=1024, ld=1024, gmax=4, B=4, dtype=sv.SV_F32, ptr=fake, ws_bytes=1 << 20):
        return L.spec_verify_token(ptr, ptr, dtype, V, ld, fake, fake, fake, gmax, fake, B, 0,
                                   None, fake, fake, gmax + 1, fake, None, None, fake, ws_bytes,
                                   None)
    assert call(V=0) == sv.SV_ERR_INVALID
    assert call(ld=1000, V=1024) == sv.SV_ERR_INVALID            # ld < V
    assert call(gmax=sv.SV_MAX_DRAFT_LEN + 1) == sv.SV_ERR_INVALID
    assert call(dtype=7) == sv.SV_ERR_INVALID
    assert call(V=1001, ld=1001, dtype=sv.SV_BF16) == sv.SV_ERR_UNSUPPORTED  # rows not 16B apart
    assert call(ptr=C.c_void_p(4098)) == sv.SV_ERR_UNSUPPORTED              # misaligned logits
    assert call(ws_bytes=16) == sv.SV_ERR_INVALID                           # workspace too small
    assert L.dspark_schedule(None, None, 4, 4, None, 2, None, None, None, None, None, None, 0,
                             None) == sv.SV_ERR_INVALID


def test_host_tensors_are_refused(sv):
    """The binding has no CPU path: tensors in host memory are refused before anything is called,
    for every entry point that computes."""
    import torch
    B, G, V = 2, 3, 64
    t = torch.zeros((B * (G + 1), V), dtype=torch.float32)
    d = torch.zeros((B * G, V), dtype=torch.float32)
    t0 = torch.arange(B, dtype=torch.int64) * (G + 1)
    d0 = torch.arange(B, dtype=torch.int64) * G
    ln = torch.full((B,), G, dtype=torch.int32)
    tok = torch.zeros(B * G, dtype=torch.int32)
    with pytest.raises((ValueError, TypeError)):
        sv.spec_verify_token(t, d, t0, d0, ln, G, tok, 0)
    with pytest.raises((ValueError, TypeError)):
        sv.spec_verify_block(t, d, t0, d0, ln, G, tok, 0)
    with pytest.raises((ValueError, TypeError)):
        sv.spec_sample_draft(d, d0, ln, G, 0)
    c = torch.full((B, G), 0.5, dtype=torch.float32)
    ml = torch.full((B,), G, dtype=torch.int32)
    sps = torch.ones(16, dtype=torch.float64)
    with pytest.raises((ValueError, TypeError)):
        sv.dspark_schedule(c, ml, sps, 15)


def test_noalloc_scratch_size_matches_header(sv):
    """The binding's SV_NOALLOC_SCRATCH_BYTES is the header's."""
    import re
    with open(sv.HEADER) as f:
        m = re.search(r"#define\s+SV_NOALLOC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", f.read())
    assert m and int(m.group(1)) << int(m.group(2)) == sv.SV_NOALLOC_SCRATCH_BYTES
