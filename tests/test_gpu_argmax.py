"""The greedy-argmax rule on the GPU: exact ties and NaN logits (GPU only).

"rvllm-metal" (section "How I know it's correct") tests the argmax with ties and NaN. The rule
here: the larger logit wins, equal logits go to the lower vocabulary index, a NaN ranks above
every number (the first NaN wins) and sets LLM_FLAG_NAN_LOGIT. Random-init logits never tie,
so the tests build the head weights on the host: two rows of the tied embedding are made equal
(exact ties) and large enough to be each sequence's maximum, or one row is NaN. Rows of the
embedding that no fed token uses only change the logits, not the hidden states.
"""
import numpy as np
import pytest

import oracle
import workloads as wl
from parity_util import check_ids, check_logits, run_gpu_teacher
from test_gpu_parity import LENGTHS, SMALL_GPT2, SMALL_LLAMA, small_workload

pytestmark = pytest.mark.gpu

# Pairs of equal head rows, one per sequence: inside one 64-column tile, across a 64-column
# partial boundary that is also a 128-column tile boundary, across a 64-column boundary inside a
# 128-column tile, and (GPT-2, vocab 1000) in the last, ragged tile.
PAIRS = {SMALL_GPT2.name: [(200, 230), (127, 128), (191, 192), (961, 999)],
         SMALL_LLAMA.name: [(200, 230), (127, 128), (191, 192), (1000, 1023)]}
BATCH_LENGTHS = np.array([5, 17, 70, 33], dtype=np.int32)


def _set_row(w, j, vals):
    row = np.asarray(vals, dtype=np.float32)
    w.tok_emb[j] = wl.f32_to_bf16_bits(row) if w.tok_emb.dtype == np.uint16 else row


def _safe_prompts(lengths, vocab, banned):
    ps = wl.draw_prompts(lengths, vocab)
    ban = set(banned)
    return [np.array([t if t not in ban else 5 for t in p], dtype=np.int32) for p in ps]


def _final_normed_hidden(m, tokens):
    """Norm_f of the last position's hidden state, from the oracle's own layer pieces."""
    pos = np.arange(len(tokens))
    h = m.embed(np.asarray(tokens), pos)
    for l in range(m.shape.n_layers):
        h, _, _ = m.layer(l, h, pos, None, None)
    return m.norm(h[-1], m.lnf_w, m.lnf_b)


def _run(shape, w, prompts, stream, variant):
    import torch
    from transformer_decoder_forward_gb300.runner import WorkloadRun
    run = WorkloadRun(small_workload(shape), host_weights=w, lengths=BATCH_LENGTHS)
    run.prompts = prompts
    run.tokens = torch.from_numpy(np.concatenate(prompts).astype(np.int32)).cuda()
    ids, z = run_gpu_teacher(run, stream, variant=variant)
    flags = run.dec.error_flags()
    run.close()
    return ids, z, flags


@pytest.mark.parametrize("variant", [0, 2, 3, 4], ids=["auto", "simt", "tcgen05", "tcgen05-swap"])
@pytest.mark.parametrize("shape", [SMALL_GPT2, SMALL_LLAMA], ids=["gpt2-f32", "llama-bf16"])
def test_exact_ties_go_to_the_lower_index(gpu_lib, shape, variant):
    if variant == 3 and shape.dtype != wl.DTYPE_BF16:
        pytest.skip("tcgen05 activation-on-M path is bf16 only")
    pairs = PAIRS[shape.name]
    banned = [j for p in pairs for j in p]
    w = wl.make_weights(shape, scale=2.0, perturb=True)
    prompts = _safe_prompts(BATCH_LENGTHS, shape.vocab, banned)
    stream = np.array([[3, 9, 44, 7]], dtype=np.int32)          # one decode step, no banned id
    m = oracle.OracleModel(w)
    # each sequence's pair gets the row c_b * (dual vector of its final normed hidden state), so
    # pair b scores c_b on sequence b and ~0 on the others; c_b clears every other logit by 5
    X = np.stack([_final_normed_hidden(m, list(prompts[b]) + [int(stream[0, b])]) for b in range(4)])
    base = np.stack([oracle.teacher_forced(m, prompts[b], stream[:, b])[-1] for b in range(4)])
    c = base.max(axis=1) + 5.0
    E = np.diag(c) @ np.linalg.pinv(X.T)                        # E_b . X_a = c_b [a == b]
    for b, (j1, j2) in enumerate(pairs):
        _set_row(w, j1, E[b])
        _set_row(w, j2, E[b])
    m = oracle.OracleModel(w)
    refs = [oracle.teacher_forced(m, prompts[b], stream[:, b]) for b in range(4)]
    for b, (j1, j2) in enumerate(pairs):
        z = refs[b][-1]
        # equal rows: equal float64 logits (up to the host BLAS's summation order)
        assert abs(z[j1] - z[j2]) <= 1e-12 * abs(z[j1]) and oracle.argmax_rule(z) in (j1, j2)
        assert z[j1] - np.delete(z, [j1, j2]).max() > 1.0
    ids, zg, flags = _run(shape, w, prompts, stream, variant)
    assert flags == 0
    for b, (j1, j2) in enumerate(pairs):
        assert zg[-1, b, j1] == zg[-1, b, j2], "equal head rows must give bitwise equal logits"
        assert int(ids[-1, b]) == j1, f"seq {b}: tie {j1}/{j2} went to {int(ids[-1, b])}"
        check_logits(zg[:, b], refs[b], shape.dtype, f"{shape.name} seq {b}")
        check_ids(ids[:1, b], refs[b][:1], f"{shape.name} seq {b} prefill")


@pytest.mark.parametrize("variant", [0, 2, 4], ids=["auto", "simt", "tcgen05-swap"])
@pytest.mark.parametrize("shape", [SMALL_GPT2, SMALL_LLAMA], ids=["gpt2-f32", "llama-bf16"])
def test_nan_logits_first_nan_wins_and_flag_is_set(gpu_lib, shape, variant):
    import transformer_decoder_forward_gb300 as L
    nan_rows = [700, 65]                       # different tiles; the lower index must win
    w = wl.make_weights(shape, scale=2.0, perturb=True)
    for j in nan_rows:
        _set_row(w, j, np.full(shape.d_model, np.nan, dtype=np.float32))
    prompts = _safe_prompts(BATCH_LENGTHS, shape.vocab, nan_rows)
    stream = np.array([[3, 9, 44, 7]], dtype=np.int32)
    m = oracle.OracleModel(w)
    ref = oracle.teacher_forced(m, prompts[0], stream[:, 0])
    assert oracle.argmax_rule(ref[-1]) == 65
    ids, zg, flags = _run(shape, w, prompts, stream, variant)
    assert flags & L.FLAG_NAN_LOGIT
    assert np.all(ids == 65), ids
    want = np.zeros(zg.shape[-1], dtype=bool)
    want[nan_rows] = True
    np.testing.assert_array_equal(np.isnan(zg), np.broadcast_to(want, zg.shape))
    assert np.all(np.isfinite(zg[..., ~want]))
