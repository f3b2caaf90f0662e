"""Launch-planning knobs against the oracle, each in a fresh process (the library reads them
once per process): with G4_GEMV_STAGED=0 and G4_GEMV_UNSPLIT_BYTES set above every
projection's size, every batch-1 projection runs on the one-slice GEMV (its GeGLU, per-layer
and argmax epilogues at E2B widths); G4_LMHEAD_STAGED=1 puts the bf16 vocabulary projection of
a staged step on the staged kernel's argmax epilogue; G4_TC_MIN_BATCH=0 keeps batch 8 on the
GEMV; and
G4_ATTN_MQA_MIN=0 keeps batch 8 on the per-head attention kernel.

Seed 1: on these shapes the fp32 oracle stays within 2e-6 of an fp64 run (some seeds do not:
seed 5 with a 20-token prompt puts the fp32 oracle itself 9e-2 from fp64 at the prefill's
last position, which no fp32 implementation can be held to)."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r'''
import json, sys
import numpy as np, torch
sys.path.insert(0, sys.argv[1])
import oracle, synth
from accelerator_decode_gb300.runtime import Decoder
sys.path.insert(0, sys.argv[1] + "/tests")
from test_gpu_decode import gpu_generate
batch = int(sys.argv[2])
cfg = synth.get_config("e2b-v8k")
w = synth.make_model_weights(cfg, "w4a16", seed=1)
prompts = synth.make_prompts(cfg["vocab"], batch, 20, seed=1)
ref = oracle.Oracle(cfg, w, max_batch=batch, max_context=64).generate(prompts, 6, keep_logits=True)
dec = Decoder(cfg, w, max_batch=batch, max_context=64)
toks, logits = gpu_generate(dec, list(prompts), 6, teacher=ref["tokens"])
err = dec.device_error()[1]
dec.close()
ok = ref["gaps"].T > 2e-3
print(json.dumps({"max_d": float(np.max(np.abs(logits - ref["logits"]))), "err": err,
                  "argmax_ok": bool(np.all((toks == ref["tokens"]) | ~ok))}))
'''


@pytest.mark.parametrize("env,batch", [
    ({"G4_GEMV_STAGED": "0", "G4_GEMV_UNSPLIT_BYTES": "1000000000000"}, 1),
    ({"G4_GEMV_STAGED": "0"}, 2),
    ({"G4_LMHEAD_STAGED": "1"}, 3),
    ({"G4_TC_MIN_BATCH": "0", "G4_ATTN_MQA_MIN": "0"}, 8),
])
def test_knob_matches_oracle(env, batch):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    e = dict(os.environ, **env)
    r = subprocess.run([sys.executable, "-c", SCRIPT, ROOT, str(batch)], env=e, capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert res["err"] == 0 and res["argmax_ok"], res
    assert res["max_d"] <= 3e-2, res
