"""The intra-GPU probes (moe_decode_megakernel_warp_gb300/probes): the source builds for
sm_103a (CPU), and on the GPU every probe reports finite positive costs with no wait
running out; the two design facts the layer kernel rests on hold on the device: a
counter handoff beats polling the data, and a loop over more straight-line code than
the instruction cache holds runs slower per instruction than one that fits."""
import math
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "..", "moe_decode_megakernel_warp_gb300", "probes", "probes.cu")


def test_probes_source_compiles(tmp_path):
    if shutil.which("nvcc") is None:
        pytest.skip("nvcc not found")
    out = tmp_path / "probes.o"
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-c", SRC, "-o", str(out)],
                   check=True)
    assert out.stat().st_size > 0


@pytest.mark.gpu
def test_probes_quick():
    from moe_decode_megakernel_warp_gb300.probes import run_probes
    res = run_probes.run("all", quick=True)
    kinds = {r["probe"] for r in res}
    assert {"acquire_load", "poll", "fence", "icache", "handoff", "clusters"} <= kinds, kinds
    cl = {r["cluster_size"]: r for r in res if r["probe"] == "clusters"}
    assert cl[1]["max_active_clusters"] >= cl[2]["max_active_clusters"] >= cl[4]["max_active_clusters"] >= 1
    for r in res:
        assert r["error"] == 0, r
        for k, v in r.items():
            if isinstance(v, float):
                assert math.isfinite(v) and v > 0, r
    hand = {(r["K"], r["mode"]): r for r in res if r["probe"] == "handoff"}
    for K in (2048, 4096):
        assert hand[(K, "counter")]["last_consumer_us_after_last_producer"] < \
            hand[(K, "poll_data")]["last_consumer_us_after_last_producer"]
    ic = next(r for r in res if r["probe"] == "icache")
    # two 96 KB blocks per pass cost more than twice one block alone (the loop no
    # longer fits the instruction cache); 96 KB + 16 KB does fit
    assert ic["two_96kb_blocks_us_per_pass"] > 2.0 * ic["alone_us_per_pass"]
