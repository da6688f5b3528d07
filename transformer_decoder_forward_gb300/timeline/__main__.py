"""python -m transformer_decoder_forward_gb300.timeline --workload NAME [--steps K] [--out CSV]"""
import argparse

from . import _child, format_report, one_step, trace


def main() -> None:
    ap = argparse.ArgumentParser(description="kernel timeline of graph-replayed decode steps")
    ap.add_argument("--workload", required=True)
    ap.add_argument("--steps", type=int, default=8)
    ap.add_argument("--out", default=None, help="CSV of the raw kernel records")
    ap.add_argument("--first", type=int, default=20, help="launches of the step to list")
    ap.add_argument("--child", action="store_true", help=argparse.SUPPRESS)
    a = ap.parse_args()
    if a.child:
        _child(a.workload, a.steps)
        return
    launches = trace(a.workload, a.steps, a.out)
    print(f"workload {a.workload}, the last complete of {a.steps} graph-replayed decode steps")
    print(format_report(one_step(launches), a.first))


if __name__ == "__main__":
    main()
