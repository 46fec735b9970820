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


def _copy_tree(tmp_path):
    """The package's csrc and the public header, in the same relative layout."""
    root = tmp_path / "repo"
    shutil.copytree(CSRC, root / "soft_capped_attention_gb300" / "csrc",
                    ignore=shutil.ignore_patterns("__pycache__"))
    shutil.copytree(os.path.join(os.path.dirname(os.path.dirname(CSRC)), "include"), root / "include")
    return root / "soft_capped_attention_gb300" / "csrc"


def test_a_kernels_tag_covers_its_own_files(tmp_path):
    d = _copy_tree(tmp_path)
    tag = lambda src: bench.files_hash(bench.kernel_files(src, str(d)), str(d))
    files = bench.kernel_files("attn_bwd_tc.cu", str(d))
    assert "attn_bwd_tc.cu" in files and "tc_common.cuh" in files and "capattn_api.cu" in files
    assert os.path.normpath("../../include/capattn.h") in files
    assert "attn_fwd1_tc.cu" not in files and "fwd_common.cuh" not in files
    dkv0, fwd0 = tag("attn_bwd_tc.cu"), tag("attn_fwd3_tc.cu")
    f = d / "attn_fwd1_tc.cu"          # another kernel's file: dK/dV's tag stays
    f.write_text(f.read_text().replace("constexpr", "constexpr ", 1) + "\nstatic int unrelated_change = 1;\n")
    assert tag("attn_bwd_tc.cu") == dkv0
    f = d / "fwd_common.cuh"           # the forwards' header: the forward's tag moves
    f.write_text(f.read_text() + "\nconstexpr int another_constant = 3;\n")
    assert tag("attn_bwd_tc.cu") == dkv0 and tag("attn_fwd3_tc.cu") != fwd0
    f = d / "tc_common.cuh"            # a header both include: both move
    f.write_text(f.read_text() + "\nconstexpr int shared_constant = 4;\n")
    assert tag("attn_bwd_tc.cu") != dkv0
