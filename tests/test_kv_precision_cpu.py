"""Why the narrow KV cache is bf16 and not fp8 (CPU, float64 oracle).

The pages' next steps name a lower-precision KV cache, fp8 among them ("rvllm-metal", "What's
basic about it": "The KV cache is F32"). What the cache stores is part of what the method
computes, so a format is usable only where the acceptance still holds: int32 ids equal wherever
the top-1/top-2 logit margin exceeds 1e-3. The oracle can store K and V rounded (its bf16 mode
rounds right after RoPE). Here the same site rounds to fp8 E4M3 instead, through torch's own
float8_e4m3fn conversion, on the batch-1 GPT-2 124M workload:
  - bf16 K/V moves the logits by a few 1e-3 and flips no id with a margin above 1e-3;
  - E4M3 K/V moves them by several 1e-2 and flips ids whose margins are well above 1e-3.
So an fp8 cache would not compute the same result under the acceptance, and is not built.
"""
import numpy as np
import pytest
import torch

import oracle
import oracle.decoder as od
import workloads as wl


def e4m3(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).to(torch.float64).numpy()


def _compare(monkeypatch, rounding):
    W = wl.WORKLOADS["gpt2-124m-fp32-b1-greedy"]
    w = wl.make_weights(W.model)
    prompt = wl.draw_prompts(W.lengths(), W.model.vocab)[0]
    stream = wl.draw_stream(1, 16, W.model.vocab)[:, 0]
    z_ref = oracle.teacher_forced(oracle.OracleModel(w), prompt, stream)
    with monkeypatch.context() as m:
        m.setattr(od, "round_bf16", rounding)
        z = oracle.teacher_forced(oracle.OracleModel(w, kv_dtype=wl.DTYPE_BF16), prompt, stream)
    top2 = np.sort(z_ref, axis=1)[:, -2:]
    margin = top2[:, 1] - top2[:, 0]
    flipped = [(float(margin[i])) for i in range(len(margin))
               if margin[i] > 1e-3 and np.argmax(z[i]) != np.argmax(z_ref[i])]
    return float(np.max(np.abs(z - z_ref))), flipped


def test_e4m3_rounding_is_torchs():
    """E4M3: 3 mantissa bits, nearest even, exponents down to 2^-6, subnormal quantum 2^-9."""
    v = np.array([1.0, 0.3, -0.3, 448.0, 2.0 ** -9, 0.06, -17.3])
    r = e4m3(v)
    assert r[0] == 1.0 and r[1] == 0.3125 and r[2] == -0.3125 and r[3] == 448.0 and r[4] == 2.0 ** -9
    assert r[5] == 15 * 2.0 ** -8 and r[6] == -18.0   # 0.06 < 2^-4: quantum 2^-8; 17.3: quantum 2


def test_bf16_kv_keeps_the_acceptance_and_fp8_kv_breaks_it(monkeypatch):
    err_bf16, flips_bf16 = _compare(monkeypatch, od.round_bf16)
    err_fp8, flips_fp8 = _compare(monkeypatch, e4m3)
    assert err_bf16 < 1e-2 and not flips_bf16
    assert err_fp8 > 3e-2 and flips_fp8 and max(flips_fp8) > 5e-3, (err_fp8, flips_fp8)
