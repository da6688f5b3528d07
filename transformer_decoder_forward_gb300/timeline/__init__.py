"""Kernel timeline of graph-replayed decode steps (a diagnostic, not part of the step).

The events around single launches serialise the kernels. The timeline instead records the
device start and end of every kernel of a normal graph-replayed step through CUPTI's activity
API, with programmatic dependent launch overlapping the kernels. A small injection library
(``ktrace.cpp``, built on first use with the CUDA toolkit's CUPTI) is loaded into a child
process through CUDA_INJECTION64_PATH. The child runs a workload's decode steps, and the
records are read back here.

A kernel's cost on the step's critical path is the time from the end of the kernel before it
to its own end ("after predecessor"). Its duration includes the time it spends launched early
and waiting on the dependency.

    python -m transformer_decoder_forward_gb300.timeline --workload gpt2-124m-fp32-b32-teacher
"""
from __future__ import annotations

import glob
import os
import re
import subprocess
import sys
from collections import OrderedDict
from typing import List, NamedTuple, Optional

_HERE = os.path.dirname(os.path.abspath(__file__))
TRACER_SRC = os.path.join(_HERE, "ktrace.cpp")
TRACER_LIB = os.path.join(_HERE, "libktrace.so")
STEP_MARKER = "k_set_args"   # every decode step's graph starts with the step-arguments node


class Launch(NamedTuple):
    start: int   # ns, device clock
    end: int
    grid: tuple
    name: str    # mangled kernel name


def cuda_home() -> str:
    return os.environ.get("CUDA_HOME", "/usr/local/cuda")


def cupti_dirs():
    """(include dir, library dir) of CUPTI in the CUDA toolkit."""
    home = cuda_home()
    inc = os.path.join(home, "include")
    for d in [os.path.join(home, "extras", "CUPTI", "lib64")] + sorted(glob.glob(os.path.join(home, "targets", "*", "lib"))):
        if glob.glob(os.path.join(d, "libcupti.so*")):
            return inc, d
    raise FileNotFoundError("libcupti.so not found under " + home)


def build_tracer() -> str:
    """Compile the injection library next to its source (once; rebuilt when the source is newer)."""
    if os.path.exists(TRACER_LIB) and os.path.getmtime(TRACER_LIB) >= os.path.getmtime(TRACER_SRC):
        return TRACER_LIB
    inc, lib = cupti_dirs()
    subprocess.run(["g++", "-shared", "-fPIC", "-O2", "-I" + inc, TRACER_SRC, "-o", TRACER_LIB, "-L" + lib, "-lcupti"],
                   check=True)
    return TRACER_LIB


def parse(path: str) -> List[Launch]:
    out = []
    with open(path) as f:
        for line in f:
            p = line.rstrip("\n").split(",", 5)
            if len(p) == 6:
                out.append(Launch(int(p[0]), int(p[1]), (int(p[2]), int(p[3]), int(p[4])), p[5]))
    out.sort()
    return out


def kernel_label(mangled: str) -> str:
    """The kernel's identifier from its mangled name: the length-prefixed k_* component. The
    length digits can follow a hash that ends in digits, so the shortest digit suffix whose
    identifier is followed by template arguments ('I') or the end of the nested name ('E') wins."""
    m = re.search(r"(\d+)(k_[A-Za-z0-9_]*)", mangled)
    if not m:
        return mangled[:40]
    digits, at = m.group(1), m.start(2)
    for j in range(len(digits) - 1, -1, -1):
        n = int(digits[j:])
        if n >= 3 and mangled[at + n: at + n + 1] in ("I", "E", ""):
            return mangled[at: at + n]
    return m.group(2)


def one_step(launches: List[Launch], which: int = -1) -> List[Launch]:
    """The launches of one step, from a step-arguments node to the next one; `which` indexes
    those bounded steps (-1: the last of them)."""
    idx = [i for i, l in enumerate(launches) if STEP_MARKER in l.name]
    if len(idx) < 2:
        raise ValueError("fewer than two steps in the trace")
    a, b = list(zip(idx[:-1], idx[1:]))[which]
    return launches[a:b]


def step_table(step: List[Launch]):
    """Per launch: (label, grid, start, end, duration, after predecessor) in microseconds, relative
    to the step's first start; and per label: launches, summed duration, summed critical-path time."""
    t0 = step[0].start
    rows, fam = [], OrderedDict()
    prev_end = t0
    for l in step:
        lab = kernel_label(l.name)
        crit = max(0, l.end - prev_end)
        rows.append((lab, l.grid, (l.start - t0) / 1e3, (l.end - t0) / 1e3, (l.end - l.start) / 1e3, crit / 1e3))
        f = fam.setdefault(lab, [0, 0.0, 0.0])
        f[0] += 1
        f[1] += (l.end - l.start) / 1e3
        f[2] += crit / 1e3
        prev_end = max(prev_end, l.end)
    return rows, fam, (prev_end - t0) / 1e3


def format_report(step: List[Launch], first: int = 20) -> str:
    rows, fam, span = step_table(step)
    out = [f"step: {len(step)} launches, {span:.1f} us from the first start to the last end", "",
           "| kernel | launches | duration (us) | on the critical path (us) |", "|---|---|---|---|"]
    for lab, (n, dur, crit) in fam.items():
        out.append(f"| {lab} | {n} | {dur:.1f} | {crit:.1f} |")
    out += ["", f"first {min(first, len(rows))} launches (us from the step's start):", "",
            "| kernel | grid | start | end | duration | after predecessor |", "|---|---|---|---|---|---|"]
    for lab, grid, s, e, d, c in rows[:first]:
        out.append(f"| {lab} | {grid[0]},{grid[1]},{grid[2]} | {s:.2f} | {e:.2f} | {d:.2f} | {c:.2f} |")
    return "\n".join(out)


def _child(workload: str, steps: int) -> None:
    """Runs inside the traced process: prefill, then `steps` graph-replayed decode steps."""
    root = os.path.dirname(os.path.dirname(_HERE))
    sys.path.insert(0, root)
    import numpy as np
    import torch
    import workloads as wl
    from transformer_decoder_forward_gb300.runner import WorkloadRun
    w = wl.WORKLOADS[workload]
    run = WorkloadRun(w, extra_steps=steps)
    run.prefill()
    torch.cuda.synchronize()
    nst = run.step_positions.shape[0]
    toks = torch.from_numpy(np.ascontiguousarray(wl.draw_stream(run.B, nst, w.model.vocab), dtype=np.int32)).cuda()
    for i in range(steps):
        run.decode(toks[i % nst], i % nst)
    torch.cuda.synchronize()
    run.close()


def trace(workload: str, steps: int = 8, out: Optional[str] = None) -> List[Launch]:
    lib = build_tracer()
    out = out or os.path.join(os.getcwd(), f"ktrace_{workload}.csv")
    _, cupti_lib = cupti_dirs()
    env = dict(os.environ, CUDA_INJECTION64_PATH=lib, KTRACE_OUT=out,
               LD_LIBRARY_PATH=cupti_lib + os.pathsep + os.environ.get("LD_LIBRARY_PATH", ""))
    subprocess.run([sys.executable, "-m", "transformer_decoder_forward_gb300.timeline", "--child", "--workload", workload,
                    "--steps", str(steps)], check=True, env=env, cwd=os.path.dirname(os.path.dirname(_HERE)))
    return parse(out)
