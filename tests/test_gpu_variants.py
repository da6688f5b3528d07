"""Model-feature variants on the GPU against the oracle: sliding-window attention, Llama 3 RoPE
scaling, Q/K norm and attention biases ("rvllm-metal", section "What the kernels do", last
paragraph), through every projection kernel and every attention kernel (GPU only)."""
from dataclasses import replace

import numpy as np
import pytest

import oracle
import workloads as wl
from parity_util import check_ids, check_logits, oracle_teacher, run_gpu_teacher
from test_gpu_parity import LENGTHS, SMALL_GPT2, SMALL_LLAMA, SMALL_LLAMA_F32, STEPS, small_workload

pytestmark = pytest.mark.gpu

# RoPE scaling chosen so that, with theta 1e4 and head_dim 64, the pairs fall in all three bands
# (wavelength below 16 kept, above 64 slowed by 4, blended in between).
ALL_FEATURES = dict(sliding_window=24, sliding_window_pattern=2, qk_norm=True, attn_bias=True,
                    rope_scaling=(4.0, 1.0, 4.0, 64), rope_theta=1e4)
VARIANT_SHAPES = [
    replace(SMALL_LLAMA, name="llama-bf16-features", **ALL_FEATURES),
    replace(SMALL_LLAMA_F32, name="llama-f32-features", **ALL_FEATURES),
    replace(SMALL_GPT2, name="gpt2-window", sliding_window=20),
]


def _cases():
    for s in VARIANT_SHAPES:
        for v in (1, 2, 3, 4):
            if v == 3 and s.dtype != wl.DTYPE_BF16:
                continue
            yield pytest.param(s, v, id=f"{s.name}-v{v}")


@pytest.mark.parametrize("shape,variant", list(_cases()))
def test_feature_variants_match_oracle(gpu_lib, shape, variant):
    from transformer_decoder_forward_gb300.runner import WorkloadRun
    w = wl.make_weights(shape, scale=2.0, perturb=True)
    model = oracle.OracleModel(w)
    run = WorkloadRun(small_workload(shape), host_weights=w, lengths=LENGTHS)
    stream = wl.draw_stream(run.B, STEPS, shape.vocab)
    ids, z = run_gpu_teacher(run, stream, variant=variant)
    assert run.dec.error_flags() == 0
    run.close()
    for b in range(run.B):
        ref = oracle_teacher(model, run.prompts[b], stream[:, b])
        check_logits(z[:, b], ref, shape.dtype, f"{shape.name} v{variant} seq {b}")
        check_ids(ids[:, b], ref, f"{shape.name} v{variant} seq {b}")


def test_window_longer_than_context_changes_nothing(gpu_lib, monkeypatch):
    """A window wider than every context gives bit-identical results to no window. Windowed
    bf16-weight models take the windowed tensor-core prefill attention; the run without a window
    is pinned to the same kernel (LLM_PREFILL_ATTN=1), so the two compute alike."""
    from transformer_decoder_forward_gb300.runner import WorkloadRun
    monkeypatch.setenv("LLM_PREFILL_ATTN", "1")
    w = wl.make_weights(SMALL_LLAMA, scale=2.0, perturb=True)
    stream = wl.draw_stream(len(LENGTHS), STEPS, SMALL_LLAMA.vocab)
    out = []
    for s in (SMALL_LLAMA, replace(SMALL_LLAMA, sliding_window=10_000)):
        run = WorkloadRun(small_workload(s), host_weights=w, lengths=LENGTHS)
        out.append(run_gpu_teacher(run, stream))
        run.close()
    np.testing.assert_array_equal(out[0][0], out[1][0])
    np.testing.assert_array_equal(out[0][1], out[1][1])
