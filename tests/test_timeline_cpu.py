"""The kernel-timeline reader on a synthetic record file (no GPU, no CUPTI)."""
import os
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
from transformer_decoder_forward_gb300 import timeline as tl  # noqa: E402

SET_ARGS = "_ZN3llm39_GLOBAL__N__6b80ab7910k_set_argsEPNS_8StepArgsES1_"
GEMM = "_ZN3llm48_GLOBAL__N__fb352e8e_15_gemm_tc_swap_cu_fa6ac76b14k_gemm_tc_swapILi32ELb1EEEvNS_12LinearParamsE"
ATTN = "_ZN3llm45_GLOBAL__N__03cf6ea6_12_attention_cu_12345678919k_attn_decode_splitIffLi1EEEvNS_16AttnDecodeParamsE"


def test_kernel_label_reads_the_length_prefixed_name():
    assert tl.kernel_label(SET_ARGS) == "k_set_args"
    assert tl.kernel_label(GEMM) == "k_gemm_tc_swap"
    assert tl.kernel_label(ATTN) == "k_attn_decode_split"


def test_one_step_and_critical_path(tmp_path):
    # two steps; in the first, the GEMM starts before the set-args node ends (overlap) and the
    # attention starts early and ends 3 us after the GEMM
    recs = [(0, 1000, SET_ARGS), (500, 5000, GEMM), (2000, 8000, ATTN),
            (10000, 11000, SET_ARGS), (10500, 14000, GEMM), (20000, 21000, SET_ARGS)]
    f = tmp_path / "k.csv"
    f.write_text("".join(f"{s},{e},1,1,1,{n}\n" for s, e, n in recs))
    launches = tl.parse(str(f))
    assert len(launches) == 6
    step = tl.one_step(launches, 0)
    assert [tl.kernel_label(l.name) for l in step] == ["k_set_args", "k_gemm_tc_swap", "k_attn_decode_split"]
    rows, fam, span = tl.step_table(step)
    assert span == pytest.approx(8.0)
    # after predecessor: set_args 1 us from the step's start, GEMM 4 us after it, attention 3 us
    assert [r[5] for r in rows] == pytest.approx([1.0, 4.0, 3.0])
    assert fam["k_attn_decode_split"][0] == 1 and fam["k_gemm_tc_swap"][1] == pytest.approx(4.5)
    last = tl.one_step(launches)
    assert [tl.kernel_label(l.name) for l in last] == ["k_set_args", "k_gemm_tc_swap"]
    assert "| k_gemm_tc_swap | 1 |" in tl.format_report(step)


def test_one_step_needs_two_markers(tmp_path):
    f = tmp_path / "k.csv"
    f.write_text(f"0,1,1,1,1,{SET_ARGS}\n")
    with pytest.raises(ValueError):
        tl.one_step(tl.parse(str(f)))
