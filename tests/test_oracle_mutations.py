"""The oracle's pins catch plausible mistakes: each case plants one mistake in a
copy of the oracle (a flipped sign, a wrong divisor, offset, index or bit
position), builds that copy, and runs the pin file that should notice; the run
must fail.  Nothing here touches the oracle in the tree or the CUDA library."""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TESTS = os.path.join(ROOT, "tests")

# (name, old text, planted text, pin file expected to fail)
MUTATIONS = [
    ("q4_k min sign", "fmaf(a, (float)get_nib(blk + 16, 32 * j + k), -bm)",
     "fmaf(a, (float)get_nib(blk + 16, 32 * j + k), bm)", "test_oracle_formats.py"),
    ("q5_k fifth bit weight", "& 1) << 4);", "& 1) << 5);", "test_oracle_formats.py"),
    ("q6_k offset", "16 * j + k) - 32);", "16 * j + k) - 31);", "test_oracle_formats.py"),
    ("q4_0 divisor", "float d32 = amax / 7.0f;", "float d32 = amax / 8.0f;", "test_oracle_formats.py"),
    ("6-bit field bit order", "    int bit = 6 * f + b;\n    if ((v >> b) & 1)",
     "    int bit = 6 * f + (5 - b);\n    if ((v >> b) & 1)", "test_oracle_formats.py"),
    ("rope rotation sign", "hv[2 * i] = a * c - b * s;", "hv[2 * i] = a * c + b * s;", "test_oracle_ops.py"),
    ("rmsnorm eps inside the root", "1.0 / sqrt(ss / (double)n + eps)", "1.0 / (sqrt(ss / (double)n) + eps)",
     "test_oracle_ops.py"),
    ("silu sign", "z / (1.0 + exp(-z))", "z / (1.0 + exp(z))", "test_oracle_ops.py"),
    ("attention scale", "1.0 / sqrt((double)head_dim)", "1.0 / (double)head_dim", "test_oracle_ops.py"),
    ("argmax tie to the highest id", "if (x[i] > x[best]) best = i;", "if (x[i] >= x[best]) best = i;",
     "test_oracle_ops.py"),
    ("gqa group map", "int gh = (int)(j / group);", "int gh = (int)(j % nkv);", "test_oracle_decode.py"),
    ("layer similarity against the update", "orc_cosine(x_in, x, h)", "orc_cosine(x_in, t, h)",
     "test_oracle_decode.py"),
]


def _mutant_tree(tmp, old, new):
    """A copy of oracle/ with one planted mistake, and the pin files beside it."""
    dst = tmp / "oracle"
    dst.mkdir()
    for f in ("__init__.py", "oracle.c", "oracle.h"):
        shutil.copy(os.path.join(ROOT, "oracle", f), dst / f)
    src = (dst / "oracle.c").read_text()
    assert src.count(old) >= 1, f"mutation target not found: {old!r}"
    (dst / "oracle.c").write_text(src.replace(old, new, 1))
    tdst = tmp / "tests"
    tdst.mkdir()
    for f in os.listdir(TESTS):
        if f.startswith("test_oracle_") or f in ("conftest.py", "blockspec.py", "inputs.py"):
            if f != os.path.basename(__file__):
                shutil.copy(os.path.join(TESTS, f), tdst / f)
    shutil.copytree(os.path.join(TESTS, "golden"), tdst / "golden")
    return tdst


@pytest.mark.parametrize("name,old,new,pins", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_fails_the_pins(tmp_path, name, old, new, pins):
    tdst = _mutant_tree(tmp_path, old, new)
    env = {k: v for k, v in os.environ.items() if k != "PYTHONPATH"}
    r = subprocess.run([sys.executable, "-m", "pytest", str(tdst / pins), "-x", "-q", "-p", "no:cacheprovider",
                        "-m", "not gpu"], cwd=str(tmp_path), env=env, capture_output=True, text=True, timeout=600)
    out = r.stdout + r.stderr
    assert "ModuleNotFoundError" not in out and "ImportError" not in out, out[-2000:]
    assert r.returncode == 1 and " failed" in out, (name, r.returncode, out[-2000:])


def test_unmutated_copy_passes_the_pins(tmp_path):
    """The harness itself: the same copy without a planted mistake passes."""
    tdst = _mutant_tree(tmp_path, "double orc_silu", "double orc_silu")
    env = {k: v for k, v in os.environ.items() if k != "PYTHONPATH"}
    r = subprocess.run([sys.executable, "-m", "pytest", str(tdst / "test_oracle_ops.py"), "-q", "-p",
                        "no:cacheprovider"], cwd=str(tmp_path), env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, (r.stdout + r.stderr)[-2000:]
