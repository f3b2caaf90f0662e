"""Parity on the five workload configurations at their stated lengths, through the C ABI.

  C1  tiny, bf16, seed 0, unit gains, 16-token prompt, 16 outputs, batch 1
  C2  E2B bf16, 128-token prompt, 512 outputs, batch 1
  C3  E2B W4A16, 128-token prompt, 512 outputs, batch 1
  C4  E2B W4A16 at batch 64, 128 + 512, four sampled sequences decoded by the oracle alone
      (sequences are independent; this is the batch-64 launch configuration at 128..639 keys)
  C5  agent replay, E2B W4A16, batch 8: a 500-token start and the first four turns (375
      appended ids after the previous turn's last output, 32 outputs each; context 2,128),
      one sampled sequence against the oracle

Decoding is teacher-forced: at every step the GPU and the oracle consume the same token (the
oracle's argmax), so every step's logits are compared ("One TPU chip, eight agents", The
engine: cached decode checked against a full re-run, token agreement only where the top-2
gap is clear).  Bars: max |logit difference| <= 3e-2 and cosine >= 0.999 at every step; the
GPU's argmax equals the oracle's wherever the oracle's top-2 gap exceeds 2e-3.  Each test
reports max |d|, min cosine and the number of near-tie steps; with G4_PARITY_REPORT set to a
path, the figures are also appended there as JSON lines.

The E2B weights are the benchmark's (synth.make_model_weights)."""
import json
import os
import time

import numpy as np
import pytest

import oracle
import synth

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
torch = pytest.importorskip("torch")

LOGIT_TOL = 3e-2
COS_MIN = 0.999
GAP_TIE = 2e-3


@pytest.fixture(scope="module")
def rt():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from accelerator_decode_gb300 import runtime
    return runtime


class Stats:
    def __init__(self, label):
        self.label, self.max_d, self.min_cos, self.steps, self.ties, self.t0 = label, 0.0, 1.0, 0, 0, time.time()

    def add(self, gpu_logits, ref_logits):
        """gpu_logits, ref_logits [n, V] for the compared sequences."""
        for g, r in zip(gpu_logits, ref_logits):
            g64, r64 = g.astype(np.float64), r.astype(np.float64)
            self.max_d = max(self.max_d, float(np.max(np.abs(g64 - r64))))
            self.min_cos = min(self.min_cos, float(g64 @ r64 / np.linalg.norm(g64) / np.linalg.norm(r64)))
            top2 = np.sort(r)[-2:]
            gap = float(top2[1] - top2[0])
            self.steps += 1
            if gap <= GAP_TIE:
                self.ties += 1
            else:
                assert int(np.argmax(g)) == int(np.argmax(r)), (self.label, self.steps, gap)
            assert self.max_d <= LOGIT_TOL, (self.label, self.steps, self.max_d)
            assert self.min_cos >= COS_MIN, (self.label, self.steps, self.min_cos)

    def report(self):
        rec = {"config": self.label, "compared_steps": self.steps, "max_abs_logit_diff": self.max_d,
               "min_cosine": self.min_cos, "near_tie_steps": self.ties, "wall_s": round(time.time() - self.t0, 1)}
        print("PARITY", json.dumps(rec))
        path = os.environ.get("G4_PARITY_REPORT")
        if path:
            with open(path, "a") as f:
                f.write(json.dumps(rec) + "\n")


def lockstep(dec, o, prompts, n_out, sample, stats):
    """Prefill every sequence on the GPU and the sampled ones in the oracle (oracle rows are
    0..len(sample)-1), then n_out - 1 decode steps teacher-forced on the oracle's argmax for
    the sampled sequences (the others feed their own argmax)."""
    B = len(prompts)
    nxt, lg = dec.prefill(list(range(B)), list(prompts), want_logits=True)
    ol = o.prefill(np.arange(len(sample)), np.asarray(prompts)[sample])
    torch.cuda.synchronize()
    stats.add(lg.cpu().numpy()[sample], ol)
    T = len(prompts[0])
    d_slots = torch.arange(B, dtype=torch.int32, device="cuda")
    pos = torch.full((B,), T, dtype=torch.int32, device="cuda")
    tok = nxt.clone()
    out = torch.empty(B, dtype=torch.int32, device="cuda")
    lgt = torch.empty(B, dec.cfg["vocab"], dtype=torch.float32, device="cuda")
    idx = torch.tensor(sample, dtype=torch.long, device="cuda")
    for s in range(1, n_out):
        forced = oracle.greedy_argmax(ol).astype(np.int32)
        tok.index_copy_(0, idx, torch.from_numpy(forced).cuda())
        dec.decode_step(d_slots, tok, pos, out, lgt)
        ol = o.step(np.arange(len(sample)), forced, np.full(len(sample), T + s - 1))
        torch.cuda.synchronize()
        stats.add(lgt[idx].cpu().numpy(), ol)
        tok.copy_(out)
        pos += 1


def test_c1_tiny_exact_config(rt):
    cfg = synth.get_config("tiny")
    w = synth.make_weights(cfg, "bf16", seed=0)          # N(0, 0.02) bf16, gains 1, lambda 1
    prompts = synth.make_prompts(cfg["vocab"], 1, 16, seed=0)
    st = Stats("C1 tiny bf16 16+16")
    dec = rt.Decoder(cfg, w, max_batch=1, max_context=32)
    lockstep(dec, oracle.Oracle(cfg, w, max_batch=1, max_context=32), list(prompts), 16, [0], st)
    assert dec.device_error()[1] == 0
    dec.close()
    # the oracle's own rounding: fp32 against fp64 over the same tokens
    ref32 = oracle.Oracle(cfg, w, max_batch=1, max_context=32).generate(prompts, 16, keep_logits=True)
    ref64 = oracle.Oracle(cfg, w, max_batch=1, max_context=32, dtype=np.float64).generate(prompts, 16,
                                                                                          keep_logits=True)
    assert np.array_equal(ref32["tokens"], ref64["tokens"])
    st.label += f" (oracle fp32 vs fp64: {np.max(np.abs(ref32['logits'] - ref64['logits'])):.2e})"
    st.report()


@pytest.mark.parametrize("fmt", ["bf16", "w4a16"])
def test_c2_c3_e2b_batch1_128_plus_512(rt, fmt):
    cfg = synth.get_config("e2b")
    w = synth.make_model_weights(cfg, fmt, seed=0)
    prompts = synth.make_prompts(cfg["vocab"], 1, 128, seed=0)
    st = Stats(f"{'C2' if fmt == 'bf16' else 'C3'} e2b {fmt} b1 128+512")
    dec = rt.Decoder(cfg, w, max_batch=1, max_context=640)
    o = oracle.Oracle(cfg, w, max_batch=1, max_context=640)
    lockstep(dec, o, list(prompts), 512, [0], st)
    assert dec.device_error()[1] == 0
    dec.close()
    st.report()


def test_c4_e2b_batch64_sampled(rt):
    cfg = synth.get_config("e2b")
    w = synth.make_model_weights(cfg, "w4a16", seed=0)
    B = 64
    prompts = synth.make_prompts(cfg["vocab"], B, 128, seed=0)
    sample = [0, 21, 42, 63]
    st = Stats("C4 e2b w4a16 b64 128+512 (4 sampled)")
    dec = rt.Decoder(cfg, w, max_batch=B, max_context=640)
    o = oracle.Oracle(cfg, w, max_batch=len(sample), max_context=640)
    lockstep(dec, o, list(prompts), 512, sample, st)
    assert dec.device_error()[1] == 0
    dec.close()
    st.report()


def test_c5_agent_replay_first_turns(rt):
    wl = synth.get_workload("e2b-w4a16-replay-b8")
    cfg = synth.get_config(wl["config"])
    w = synth.make_model_weights(cfg, wl["fmt"], seed=0)
    B, turns = wl["batch"], 4
    sched = synth.replay_schedule(start=wl["prompt"], end=wl["prompt"] + wl["turns"] * wl["turn_append"],
                                  turns=wl["turns"], outputs=wl["out"])[:turns + 1]
    max_ctx = sched[0][0] + sum(a + o for a, o in sched[1:]) + 64
    st = Stats(f"C5 replay e2b w4a16 b8, {turns} turns (seq 0)")
    dec = rt.Decoder(cfg, w, max_batch=B, max_context=max_ctx)
    o = oracle.Oracle(cfg, w, max_batch=1, max_context=max_ctx)
    d_slots = torch.arange(B, dtype=torch.int32, device="cuda")
    tok = torch.empty(B, dtype=torch.int32, device="cuda")
    out = torch.empty(B, dtype=torch.int32, device="cuda")
    lgt = torch.empty(B, cfg["vocab"], dtype=torch.float32, device="cuda")
    ctx, last = 0, None
    for turn, (fresh, outs) in enumerate(sched):
        ids = synth.make_prompts(cfg["vocab"], B, fresh, seed=1000 + turn)
        if last is not None:
            ids = np.concatenate([last[:, None], ids], axis=1)
        nxt, lg = dec.prefill(list(range(B)), list(ids), start_pos=[ctx] * B, want_logits=True)
        ol = o.prefill([0], ids[:1], start_pos=[ctx])
        torch.cuda.synchronize()
        ctx += ids.shape[1]
        if outs == 0:
            continue
        st.add(lg.cpu().numpy()[:1], ol)
        tok.copy_(nxt)
        pos = torch.full((B,), ctx, dtype=torch.int32, device="cuda")
        for s in range(outs - 1):
            forced = oracle.greedy_argmax(ol).astype(np.int32)
            tok[0] = int(forced[0])
            dec.decode_step(d_slots, tok, pos, out, lgt)
            ol = o.step([0], forced, [ctx + s])
            torch.cuda.synchronize()
            st.add(lgt[:1].cpu().numpy(), ol)
            tok.copy_(out)
            pos += 1
        last_forced = oracle.greedy_argmax(ol).astype(np.int32)
        last = out.cpu().numpy().astype(np.int32)
        last[0] = last_forced[0]
        ctx += outs - 1
    assert dec.device_error()[1] == 0
    dec.close()
    st.report()
