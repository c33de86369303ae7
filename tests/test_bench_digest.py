"""The kernel-source digest that ties the benchmark's recorded DRAM traffic
to the sources it was captured on: comments and whitespace do not change it,
code does (CPU only)."""
import os
import shutil

import bench

CSRC = os.path.join(bench.ROOT, "verify_matvec_gb300", "csrc")


def _copy(tmp_path):
    d = tmp_path / "csrc"
    shutil.copytree(CSRC, d)
    return d


def _edit(d, name, old, new):
    p = d / name
    text = p.read_text()
    assert old in text
    p.write_text(text.replace(old, new, 1))


def test_comments_and_whitespace_keep_the_digest(tmp_path):
    d = _copy(tmp_path)
    base = bench.source_digest(str(d))
    assert base == bench.source_digest(CSRC)
    _edit(d, "cbq_kernels.cu", "namespace cbq {", "// a new comment\n/* and a block\n   comment */\nnamespace   cbq {")
    assert bench.source_digest(str(d)) == base


def test_code_changes_the_digest(tmp_path):
    d = _copy(tmp_path)
    base = bench.source_digest(str(d))
    _edit(d, "cbq_kernels.cu", "constexpr int kMinStages = 4;", "constexpr int kMinStages = 3;")
    assert bench.source_digest(str(d)) != base


def test_string_literals_are_code(tmp_path):
    """A '//' inside a string literal is not a comment."""
    d = _copy(tmp_path)
    (d / "extra.h").write_text('const char *a = "x // y";\n')
    one = bench.source_digest(str(d))
    (d / "extra.h").write_text('const char *a = "x // z";\n')
    assert bench.source_digest(str(d)) != one


def test_other_translation_units_do_not_change_it(tmp_path):
    """The digest follows the profiled kernels' translation unit and the
    headers only: a code change in another translation unit keeps it."""
    d = _copy(tmp_path)
    base = bench.source_digest(str(d))
    _edit(d, "cbq_mmq.cu", "constexpr int kM2Stages = 2;", "constexpr int kM2Stages = 3;")
    assert bench.source_digest(str(d)) == base
    _edit(d, "cbq_pipe.cuh", "struct Producer {", "struct Producer { int unused_ = 0;")
    assert bench.source_digest(str(d)) != base
