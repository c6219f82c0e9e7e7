"""The product (the package and its CUDA sources) never reaches the oracle, and it
fails loudly, with no fallback, when its library cannot be built or loaded."""
import os
import re
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "moe_decode_megakernel_warp_gb300")


def test_no_product_source_imports_or_includes_the_oracle():
    pat = re.compile(r"^\s*(import\s+oracle|from\s+oracle|#\s*include\s+[\"<][^\">]*oracle)", re.M)
    for dirpath, _, files in os.walk(PKG):
        if "_build" in dirpath:
            continue
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                src = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert not pat.search(src), os.path.join(dirpath, f)


def test_loading_the_product_leaves_the_oracle_unloaded():
    code = ("import sys; sys.path.insert(0, %r); import moe_decode_megakernel_warp_gb300 as m; m.lib(); "
            "print('oracle' in sys.modules)" % ROOT)
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr
    assert out.stdout.strip().splitlines()[-1] == "False"


def test_every_entry_point_raises_when_the_library_cannot_be_built():
    code = ("import sys; sys.path.insert(0, %r)\n"
            "import moe_decode_megakernel_warp_gb300 as m\n"
            "def no_build(*a, **k): raise RuntimeError('nvcc failed')\n"
            "m.build = no_build\n"
            "m._LIB = None\n"
            "calls = [lambda: m.msm_sync(None), lambda: m.msm_accept(None, 0, [0]*16, list(range(-1, 15)), 0, [0], [0], 0),\n"
            "         lambda: m.msm_verify_step(None, 0, list(range(-1, 15)), 0, [0], [0], 0, 0)]\n"
            "n = 0\n"
            "for c in calls:\n"
            "    try:\n"
            "        c()\n"
            "    except RuntimeError as e:\n"
            "        n += 'nvcc failed' in str(e)\n"
            "print(n)\n" % ROOT)
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr
    assert out.stdout.strip().splitlines()[-1] == "3"
