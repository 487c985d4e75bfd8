"""The allocation-free chain verify, for callers that cannot allocate device
memory (their host program owns every allocation, or their memory budget is
fixed at start-up): sv_verify_chain_noalloc must give the same results as
sv_verify_chain with a caller workspace, on consecutive calls that share the
library's static scratch, on a request that fills the scratch to its last
byte, and through the Python wrapper with no draft positions.  Collected last
on purpose."""
import ctypes as C

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _ptr(t):
    return C.c_void_p(t.data_ptr()) if t is not None else None


def _outputs(B, N, dev):
    return dict(tokens=torch.full((B, N + 1), -7, dtype=torch.int32, device=dev),
                accept_len=torch.full((B,), -7, dtype=torch.int32, device=dev),
                q_prob=torch.zeros(B, max(N, 1), device=dev),
                p_prob=torch.zeros(B, max(N, 1), device=dev),
                margin=torch.zeros(B, N + 1, device=dev),
                status=torch.full((B,), 77, dtype=torch.int32, device=dev))


def test_noalloc_matches_workspace_entry_point():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_vocab_gb300 as sv
    from speculative_decoding_verification_vocab_gb300 import synth
    lib = sv.load_library()
    dev = torch.device("cuda:0")
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    cases = [(torch.bfloat16, 24, 5, 32000, 1.0, 0), (torch.float32, 7, 3, 5003, 0.8, 1)]
    for dtype, B, N, V, T, seed in cases:
        cfg = synth.Config(98, "noalloc", "chain", B=B, V=V, dtype=dtype, sigma_q=3.0, N=N,
                           sigma_noise=0.4, temperature=T)
        for call in range(2):                       # two calls in a row share the scratch
            vq, dp, d = synth.chain_inputs(cfg, seed=seed * 10 + call, device=dev)
            ref = sv.verify_chain(vq, dp, d, temperature=T, seed=5, step=call)
            out = _outputs(B, N, dev)
            st = lib.sv_verify_chain_noalloc(
                _ptr(vq), _ptr(dp), sv.SV_BF16 if dtype == torch.bfloat16 else sv.SV_F32,
                _ptr(d), B, N, V, T, 5, call, _ptr(out["tokens"]), _ptr(out["accept_len"]),
                _ptr(out["q_prob"]), _ptr(out["p_prob"]), _ptr(out["margin"]),
                _ptr(out["status"]), stream, None)
            assert st == sv.SV_OK, lib.sv_last_error()
            torch.cuda.synchronize()
            for k in ("tokens", "accept_len", "status"):
                assert torch.equal(out[k], ref[k]), k
            for k in ("q_prob", "p_prob"):
                err = (out[k][:, :N] - ref[k][:, :N]).abs().max().item() if N else 0.0
                assert err <= 1e-6, (k, err)
            assert torch.allclose(out["margin"], ref["margin"], atol=2e-6, equal_nan=True)


def test_noalloc_rejects_requests_beyond_its_scratch():
    import speculative_decoding_verification_vocab_gb300 as sv
    lib = sv.load_library()
    cap = lib.sv_verify_chain_noalloc_max_bytes()
    B, N, V = 16384, 7, 128256
    assert lib.sv_verify_chain_workspace(B, N, V) > cap
    # valid pointers (the argument checks come first); the call refuses
    # before it reads or writes any of them
    held = torch.zeros(64, dtype=torch.int32, device="cuda:0")
    buf = _ptr(held)
    st = lib.sv_verify_chain_noalloc(buf, buf, sv.SV_BF16, buf, B, N, V, 1.0, 0, 0, buf,
                                     buf, None, None, None, buf, None, None)
    assert st == sv.SV_ERR_UNSUPPORTED
    msg = lib.sv_last_error().decode()
    assert "static scratch" in msg and str(cap) in msg


def _compare(out, ref, N):
    for k in ("tokens", "accept_len", "status"):
        assert torch.equal(out[k], ref[k]), k
    for k in ("q_prob", "p_prob"):
        err = (out[k][:, :N] - ref[k][:, :N]).abs().max().item() if N else 0.0
        assert err <= 1e-6, (k, err)
    assert torch.allclose(out["margin"], ref["margin"], atol=2e-6, equal_nan=True)


def test_noalloc_at_full_scratch_and_through_the_wrapper():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_vocab_gb300 as sv
    from speculative_decoding_verification_vocab_gb300 import synth
    lib = sv.load_library()
    dev = torch.device("cuda:0")
    cap = lib.sv_verify_chain_noalloc_max_bytes()
    # the largest batch of large-vocabulary chains whose workspace fits: the
    # last regions of the static array are used
    N, V = 7, 128256
    B = max(b for b in range(1, 4096) if lib.sv_verify_chain_workspace(b, N, V) <= cap)
    assert lib.sv_verify_chain_workspace(B + 1, N, V) > cap
    cfg = synth.Config(97, "noalloc_full", "chain", B=B, V=V, dtype=torch.bfloat16, sigma_q=3.0,
                       N=N, sigma_noise=0.255)
    vq, dp, d = synth.chain_inputs(cfg, seed=3, device=dev)
    ref = sv.verify_chain(vq, dp, d, temperature=1.0, seed=9, step=4)
    out = _outputs(B, N, dev)
    sv.sv_verify_chain_noalloc(vq, dp, d, 1.0, 9, 4, out["tokens"], out["accept_len"],
                               out["q_prob"], out["p_prob"], out["margin"], out["status"])
    torch.cuda.synchronize()
    _compare(out, ref, N)
    del vq, dp, d
    # N = 0 through the wrapper: no draft rows or tokens, a bonus draw only
    cfg = synth.Config(96, "noalloc_bonus", "chain", B=5, V=1000, dtype=torch.float32,
                       sigma_q=2.0, N=0, sigma_noise=0.5)
    for call in range(2):
        vq, dp, d = synth.chain_inputs(cfg, seed=call, device=dev)
        ref = sv.verify_chain(vq, None, None, temperature=1.0, seed=2, step=call)
        out = _outputs(5, 0, dev)
        sv.sv_verify_chain_noalloc(vq, None, None, 1.0, 2, call, out["tokens"],
                                   out["accept_len"], out["q_prob"], out["p_prob"],
                                   out["margin"], out["status"])
        torch.cuda.synchronize()
        _compare(out, ref, 0)
        assert out["accept_len"].eq(0).all()
