"""bench.py tags the ncu traffic figures with a hash of the kernel sources'
code: editing a comment or whitespace keeps it, any code change alters it,
and directories in the source folder are skipped."""

import os
import shutil
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import bench  # noqa: E402

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "soft_capped_attention_gb300", "csrc")


def _copy(tmp_path):
    dst = tmp_path / "csrc"
    shutil.copytree(CSRC, dst, ignore=shutil.ignore_patterns("__pycache__"))
    return dst


def test_comments_and_whitespace_keep_the_hash(tmp_path):
    d = _copy(tmp_path)
    h0 = bench.kernel_source_hash(str(d))
    f = d / "prepass.cu"
    f.write_text(f.read_text() + "\n// a trailing comment\n/* and a block\n   comment */\n   \n")
    (d / "__pycache__").mkdir()
    assert bench.kernel_source_hash(str(d)) == h0


def test_code_changes_alter_the_hash(tmp_path):
    d = _copy(tmp_path)
    h0 = bench.kernel_source_hash(str(d))
    f = d / "fwd_common.cuh"
    src = f.read_text()
    assert "constexpr float kTopMax = 100.0f;" in src
    f.write_text(src.replace("constexpr float kTopMax = 100.0f;", "constexpr float kTopMax = 99.0f;"))
    assert bench.kernel_source_hash(str(d)) != h0
