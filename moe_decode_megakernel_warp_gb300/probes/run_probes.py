"""Build and run the intra-GPU probes of probes.cu (one JSON object per result).

    python -m moe_decode_megakernel_warp_gb300.probes.run_probes [poll|fence|icache|handoff|clusters|all] [--quick]

The probes measure, on the current GPU, the costs the layer kernel's handoff and
prefetch design rests on: GPU-scope acquire-poll latency (idle and with bulk copies
in flight), the cost of a gpu-scope fence (idle, after stores, with bulk copies in
flight), instruction-cache capacity (straight-line code blocks run in a loop), a
grid-wide handoff polled element by element against one behind a counter, and how many
clusters of the layer kernel's block shape fit on the GPU at once.
"""
import json
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "probes.cu")
EXE = os.path.join(HERE, "_build", "probes")


def build(force=False):
    """Compile probes.cu for sm_103a (once); returns the executable's path."""
    if not force and os.path.exists(EXE) and os.path.getmtime(EXE) >= os.path.getmtime(SRC):
        return EXE
    os.makedirs(os.path.dirname(EXE), exist_ok=True)
    cmd = ["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-o", EXE, SRC]
    subprocess.run(cmd, check=True)
    return EXE


def run(which="all", quick=False, timeout=300):
    """Run the probes; returns the list of result dicts. Raises if a probe's wait ran out."""
    args = [build(), which] + (["--quick"] if quick else [])
    p = subprocess.run(args, capture_output=True, text=True, timeout=timeout)
    results = [json.loads(line) for line in p.stdout.splitlines() if line.startswith("{")]
    if p.returncode != 0:
        raise RuntimeError("probes failed (exit %d): %s" % (p.returncode, p.stderr.strip()[-500:]))
    return results


def main(argv=None):
    argv = sys.argv[1:] if argv is None else argv
    which = next((a for a in argv if not a.startswith("--")), "all")
    for r in run(which, quick="--quick" in argv):
        print(json.dumps(r))


if __name__ == "__main__":
    main()
