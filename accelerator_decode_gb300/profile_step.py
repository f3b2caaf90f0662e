"""Run a few decode steps of a synthetic model at a chosen context length, for a profiler.

    python -m accelerator_decode_gb300.profile_step --config e2b-v8k --fmt w4a16 \
        --batch 64 --position 639 --steps 3

No prefill: every sequence decodes at `position` over a cache that holds zeros below it.
The kernels do the same work as after a real prompt of that length (attention reads
position + 1 keys of every layer's window; no launch depends on the cache's values), so a
profiler sees the launch configuration and the bytes of a step at that context without the
hundreds of prefill launches a real prompt would add in front of it.  Prints the CUDA-event
time of each step.
"""
import argparse
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import synth  # noqa: E402
from accelerator_decode_gb300.runtime import Decoder  # noqa: E402


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--config", default="e2b-v8k", choices=sorted(synth.CONFIGS))
    ap.add_argument("--fmt", default="w4a16", choices=["bf16", "w4a16"])
    ap.add_argument("--tables", default="bf16", choices=["bf16", "int4"])
    ap.add_argument("--kv", default="bf16", choices=["bf16", "int8"])
    ap.add_argument("--batch", type=int, default=1)
    ap.add_argument("--position", type=int, default=128)
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--phases", action="store_true", help="also time every phase (direct launches)")
    a = ap.parse_args(argv)
    cfg = synth.get_config(a.config)
    w = synth.make_model_weights(cfg, a.fmt, seed=a.seed, tables=a.tables)
    ctx = ((a.position + 1 + 63) // 64) * 64
    dec = Decoder(cfg, w, max_batch=a.batch, max_context=ctx, kv_format=a.kv)
    del w
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        slots = torch.arange(a.batch, dtype=torch.int32, device="cuda")
        tok = torch.from_numpy(synth.make_prompts(cfg["vocab"], a.batch, 1, seed=a.seed)[:, 0].copy()).cuda()
        pos = torch.full((a.batch,), a.position, dtype=torch.int32, device="cuda")
        out = torch.empty(a.batch, dtype=torch.int32, device="cuda")
        for i in range(a.steps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            dec.decode_step(slots, tok, pos, out, None, stream=st)
            e1.record(st)
            e1.synchronize()
            print(f"step {i}: {e0.elapsed_time(e1) * 1e3:.1f} us", flush=True)
        if a.phases:
            prof = dec.profile_step(slots, tok, pos, out, None, repeats=2, stream=st)
            for ph in prof:
                print(f"phase {ph['name']:24s} launches {ph['launches'] // 2:4d}  {ph['ms_total'] / 2 * 1e3:9.1f} us/step",
                      flush=True)
        status, word = dec.device_error(stream=st)
    dec.close()
    if word:
        print(f"device error word {word}", file=sys.stderr)
        return 1
    return 0


if __name__ == "__main__":
    sys.exit(main())
