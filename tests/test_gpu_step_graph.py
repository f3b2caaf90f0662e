"""The decode step as the benchmark runs it.  On a non-default stream g4_decode_step replays
a captured CUDA graph (captured on the first call, re-captured when n_seq or the pointer set
changes); on the legacy default stream, where the other decode tests run, it launches the
kernels directly.  Both must give the same ids and logits bit for bit, and match the oracle."""
import numpy as np
import pytest

import oracle
import synth
from test_gpu_decode import check_parity, gpu_generate

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def rt():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from accelerator_decode_gb300 import runtime
    return runtime


@pytest.mark.parametrize("mode", [0, 1])
def test_graph_replay_equals_direct_launches_and_oracle(rt, mode):
    cfg = synth.get_config("tiny10")
    w = synth.make_weights(cfg, "w4a16", seed=31, gain_std=0.1, layer_scale_std=0.05)
    prompts = synth.make_prompts(cfg["vocab"], 2, 12, seed=10)
    ref = oracle.Oracle(cfg, w, max_batch=2, max_context=48).generate(prompts, 10, keep_logits=True)
    direct = rt.Decoder(cfg, w, max_batch=2, max_context=48)
    direct.set_step_mode(mode)
    t0, l0 = gpu_generate(direct, list(prompts), 10)
    assert direct.device_error()[1] == 0
    direct.close()
    graph = rt.Decoder(cfg, w, max_batch=2, max_context=48)
    graph.set_step_mode(mode)
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        t1, l1 = gpu_generate(graph, list(prompts), 10)
        assert graph.device_error(stream=st)[1] == 0
    torch.cuda.synchronize()
    graph.close()
    np.testing.assert_array_equal(t0, t1)
    np.testing.assert_array_equal(l0, l1)
    def rerun(teacher):
        d = rt.Decoder(cfg, w, max_batch=2, max_context=48)
        d.set_step_mode(mode)
        with torch.cuda.stream(st):
            r = gpu_generate(d, list(prompts), 10, teacher=teacher)
        torch.cuda.synchronize()
        d.close()
        return r

    check_parity(ref, t1, l1, f"graph replay/mode {mode}", rerun=rerun)
