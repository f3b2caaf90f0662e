"""Parity at E2B scale (full widths, 262,144 vocab) and at long contexts with E2B head dims.

E2B: both weight formats, a short prompt and a few greedy steps, compared with the oracle.
mid: E2B's head dims (256 / 512), window 512 and 8 query heads on a narrow model, prefilled
past the window (700 tokens) so the sliding window binds, full layers split over many key
chunks, and K/V tiles are pipelined."""
import numpy as np
import pytest

import oracle
import synth
from test_gpu_decode import COS_MIN, GAP_TIE, LOGIT_TOL, _cos, gpu_generate

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def rt():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from accelerator_decode_gb300 import runtime
    return runtime


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("fmt", ["w4a16", "bf16"])
def test_e2b_short_decode(rt, fmt, mode):
    cfg = synth.get_config("e2b")
    w = synth.make_model_weights(cfg, fmt, seed=0)
    prompts = synth.make_prompts(cfg["vocab"], 1, 24, seed=0)
    ref = oracle.Oracle(cfg, w, max_batch=1, max_context=64).generate(prompts, 8, keep_logits=True)
    dec = rt.Decoder(cfg, w, max_batch=1, max_context=64)
    dec.set_step_mode(mode)
    assert dec.step_mode(1) == mode
    toks, logits = gpu_generate(dec, list(prompts), 8, teacher=ref["tokens"])
    assert dec.device_error()[1] == 0
    dec.close()
    err = np.max(np.abs(logits - ref["logits"]))
    assert err <= LOGIT_TOL, err
    assert min(_cos(logits[s][0], ref["logits"][s][0]) for s in range(8)) >= 0.999
    ok = ref["gaps"].T > GAP_TIE
    assert np.all((toks == ref["tokens"]) | ~ok)


@pytest.mark.parametrize("batch", [1, 3])
def test_long_context_e2b_heads(rt, batch):
    cfg = synth.get_config("mid")
    w = synth.make_weights(cfg, "w4a16", seed=4, gain_std=0.1)
    prompts = synth.make_prompts(cfg["vocab"], batch, 700, seed=8)
    ref = oracle.Oracle(cfg, w, max_batch=batch, max_context=768).generate(prompts, 6, keep_logits=True)
    dec = rt.Decoder(cfg, w, max_batch=batch, max_context=768)
    toks, logits = gpu_generate(dec, list(prompts), 6, teacher=ref["tokens"])
    assert dec.device_error()[1] == 0
    dec.close()
    assert np.max(np.abs(logits - ref["logits"])) <= LOGIT_TOL
    ok = ref["gaps"].T > GAP_TIE
    assert np.all((toks == ref["tokens"]) | ~ok)


def test_e2b_batch64_sampled_sequences(rt):
    """The batch-64 workload's launch configuration (tensor-core GEMMs, 64 sequences per step)
    at E2B size.  Sequences are independent, so the oracle decodes a sample of them alone;
    every sampled sequence's logits must match, teacher-forced on the oracle's tokens."""
    cfg = synth.get_config("e2b")
    w = synth.make_model_weights(cfg, "w4a16", seed=0)
    B, T, n_out = 64, 8, 3
    prompts = synth.make_prompts(cfg["vocab"], B, T, seed=3)
    sample = [0, 17, 42, 63]
    ref = oracle.Oracle(cfg, w, max_batch=len(sample), max_context=32).generate(prompts[sample], n_out,
                                                                                keep_logits=True)
    teacher = np.zeros((B, n_out), np.int32)
    teacher[sample] = ref["tokens"]
    dec = rt.Decoder(cfg, w, max_batch=B, max_context=32)
    toks, logits = gpu_generate(dec, list(prompts), n_out, teacher=teacher)
    assert dec.device_error()[1] == 0
    dec.close()
    got = logits[:, sample]
    assert np.max(np.abs(got - ref["logits"])) <= LOGIT_TOL
    assert min(_cos(got[s][i], ref["logits"][s][i]) for s in range(n_out) for i in range(len(sample))) >= COS_MIN
    ok = ref["gaps"].T > GAP_TIE
    assert np.all((toks[sample] == ref["tokens"]) | ~ok)
