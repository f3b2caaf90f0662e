"""Failure detection without a GPU fault: a bounded device wait that runs out, and an
injected allocation failure during g4_create.

The probe waits (one warp, %globaltimer-bounded) on a device flag that nothing sets; its
timeout must reach the host as G4_ERR_TIMEOUT through g4_get_device_error, and the handle must
keep decoding correctly afterwards.  The allocation hook (G4_FAIL_ALLOC_AT=n) fails the n-th
device allocation of g4_create: the call must return G4_ERR_OOM and give every byte back."""
import ctypes

import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def rt():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from accelerator_decode_gb300 import runtime
    return runtime


def _decode(dec, prompts, n_out, teacher):
    from test_gpu_decode import gpu_generate
    return gpu_generate(dec, list(prompts), n_out, teacher=teacher)


def test_timeout_probe_reports_and_handle_survives(rt):
    from accelerator_decode_gb300 import g4
    cfg = synth.get_config("tiny")
    w = synth.make_weights(cfg, "bf16", seed=3)
    prompts = synth.make_prompts(cfg["vocab"], 1, 8, seed=3)
    ref = oracle.Oracle(cfg, w, max_batch=1, max_context=32).generate(prompts, 6, keep_logits=True)
    dec = rt.Decoder(cfg, w, max_batch=1, max_context=32)
    _decode(dec, prompts, 6, ref["tokens"])
    assert dec.device_error() == (g4.G4_OK, 0)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert g4.lib.g4_timeout_probe(dec.h, stream, 20_000_000) == g4.G4_OK     # 20 ms
    status, word = dec.device_error()
    assert status == g4.G4_ERR_TIMEOUT and word & g4.G4_DEV_TIMEOUT
    assert dec.device_error() == (g4.G4_OK, 0)                             # read clears it
    assert g4.lib.g4_timeout_probe(dec.h, stream, -1) == g4.G4_ERR_INVALID_ARG
    # the context and the handle still work: a fresh run matches the oracle
    dec.release(0)
    toks, logits = _decode(dec, prompts, 6, ref["tokens"])
    assert dec.device_error() == (g4.G4_OK, 0)
    assert np.max(np.abs(logits - ref["logits"])) <= 3e-2
    dec.close()


def test_allocation_failure_returns_oom_and_frees_everything(rt, monkeypatch):
    from accelerator_decode_gb300 import g4
    cfg = synth.get_config("tiny10")
    w = synth.make_weights(cfg, "w4a16", seed=2)
    dec = rt.Decoder(cfg, w, max_batch=2, max_context=64)   # warm: context, streams, attributes
    dec.close()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    free0 = torch.cuda.mem_get_info()[0]
    hit = 0
    for n in (1, 2, 9, 40, 10_000):
        monkeypatch.setenv("G4_FAIL_ALLOC_AT", str(n))
        try:
            d = rt.Decoder(cfg, w, max_batch=2, max_context=64)
        except g4.G4Error as e:
            assert e.status == g4.G4_ERR_OOM, (n, e.status)
            hit += 1
        else:
            assert n == 10_000, "fewer allocations than expected"
            d.close()
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        free = torch.cuda.mem_get_info()[0]
        assert abs(free - free0) <= 4 << 20, (n, free0 - free)
    assert hit == 4
    monkeypatch.delenv("G4_FAIL_ALLOC_AT")
    prompts = synth.make_prompts(cfg["vocab"], 1, 8, seed=1)
    ref = oracle.Oracle(cfg, w, max_batch=1, max_context=64).generate(prompts, 4, keep_logits=True)
    d = rt.Decoder(cfg, w, max_batch=2, max_context=64)
    toks, logits = _decode(d, prompts, 4, ref["tokens"])
    d.close()
    assert np.max(np.abs(logits - ref["logits"])) <= 3e-2
