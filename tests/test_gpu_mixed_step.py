"""Mixed passes through llm_step: decode rows, new prompts and prompt chunks in one batch,
against the float64 oracle's cached sequences (GPU only)."""
from dataclasses import replace

import numpy as np
import pytest

import oracle
import workloads as wl
from parity_util import check_ids, check_logits
from test_gpu_parity import SMALL, small_workload

pytestmark = pytest.mark.gpu

# Per call: (sequence, tokens fed). A sequence continues where its previous call stopped.
CALLS = [
    [(0, 17), (1, 33), (3, 32)],             # prompts
    [(0, 1), (1, 1), (2, 40), (3, 20)],      # two decode rows first (split-K decode attention),
                                             # a new prompt, a prompt's second chunk
    [(2, 1), (3, 3), (0, 1)],                # a decode row first, a 3-token chunk, another decode row
    [(1, 90), (0, 1)],                       # a 90-token chunk (two 64-row tiles for fp32 weights), a decode row
]


WINDOWED = [replace(SMALL[2], name="small-llama-window", sliding_window=24, qk_norm=True),
            replace(SMALL[0], name="small-gpt2-window", sliding_window=20)]


@pytest.mark.parametrize("kv", [wl.DTYPE_F32, wl.DTYPE_BF16], ids=["kv-f32", "kv-bf16"])
@pytest.mark.parametrize("shape", SMALL + WINDOWED, ids=[s.name for s in SMALL + WINDOWED])
def test_mixed_step_matches_oracle(gpu_lib, shape, kv):
    import torch
    from transformer_decoder_forward_gb300.runner import WorkloadRun
    w = wl.make_weights(shape, scale=2.0, perturb=True)
    model = oracle.OracleModel(w, kv_dtype=kv)
    total = {}
    for call in CALLS:
        for b, n in call:
            total[b] = total.get(b, 0) + n
    lengths = np.array([total[b] for b in range(4)], dtype=np.int32)
    run = WorkloadRun(replace(small_workload(shape), decode_steps=0, kv_dtype=kv), host_weights=w,
                      lengths=lengths, max_prefill_tokens=256)
    streams = wl.draw_prompts(lengths, shape.vocab, seed=7)   # every token each sequence will feed
    seqs = [oracle.Sequence(model) for _ in range(4)]
    fed = [0] * 4
    for call in CALLS:
        toks, lens, starts, rows = [], [], [], []
        for b, n in call:
            toks.append(streams[b][fed[b]: fed[b] + n])
            lens.append(n)
            starts.append(fed[b])
            rows.append(b)
        tables = run.tables[torch.tensor(rows, device="cuda")].contiguous()
        tok = torch.from_numpy(np.concatenate(toks).astype(np.int32)).cuda()
        ids = torch.zeros(len(call), dtype=torch.int32, device="cuda")
        z = torch.empty((len(call), shape.vocab), dtype=torch.float32, device="cuda")
        with torch.cuda.stream(run.stream):
            run.dec.step(tok, lens, starts, tables, ids, z)
        torch.cuda.synchronize()
        assert run.dec.error_flags() == 0
        zg, ig = z.cpu().numpy(), ids.cpu().numpy()
        for i, (b, n) in enumerate(call):
            ref = seqs[b].feed(streams[b][fed[b]: fed[b] + n])        # logits after the last new token
            what = f"{shape.name} call {CALLS.index(call)} seq {b} ({n} tokens from {fed[b]})"
            check_logits(zg[i:i + 1], ref, shape.dtype, what)
            check_ids(ig[i:i + 1], ref, what)
            fed[b] += n
    run.close()


def test_prefill_is_a_step_from_position_zero(gpu_lib):
    """llm_prefill and llm_step with every start at 0 give bit-identical results."""
    import torch
    from transformer_decoder_forward_gb300.runner import WorkloadRun
    shape = SMALL[2]
    w = wl.make_weights(shape, scale=2.0, perturb=True)
    lengths = np.array([5, 17, 70], dtype=np.int32)
    out = []
    for use_step in (False, True):
        run = WorkloadRun(small_workload(shape), host_weights=w, lengths=lengths)
        z = torch.empty((3, shape.vocab), dtype=torch.float32, device="cuda")
        with torch.cuda.stream(run.stream):
            if use_step:
                run.dec.step(run.tokens, list(lengths), [0, 0, 0], run.tables, run.next_ids, z)
            else:
                run.dec.prefill(run.tokens, list(lengths), run.tables, run.next_ids, z)
        torch.cuda.synchronize()
        out.append((z.cpu().numpy(), run.next_ids.cpu().numpy()))
        run.close()
    np.testing.assert_array_equal(out[0][0], out[1][0])
    np.testing.assert_array_equal(out[0][1], out[1][1])
