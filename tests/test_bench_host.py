"""Host-side pieces of bench.py that need no GPU."""

import os
import shutil

import bench


def test_kernel_hash_ignores_comments_but_not_code(tmp_path, monkeypatch):
    """The DRAM counters in profiles/traffic.json stay attached to the code
    through comment edits, and are dropped by any change to the code."""
    csrc = tmp_path / "sparse_attention_top_expand_gb300" / "csrc"
    csrc.mkdir(parents=True)
    src = os.path.join(bench.ROOT, "sparse_attention_top_expand_gb300", "csrc")
    for name in bench.KERNEL_SOURCES:
        shutil.copy(os.path.join(src, name), csrc / name)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    base = bench.kernel_source_hash()
    k = csrc / "smq_kernels.cuh"
    text = k.read_text()
    k.write_text("// a new comment\n/* and a block\n   comment */\n" + text.replace("\n", "\n\n", 3))
    assert bench.kernel_source_hash() == base
    k.write_text(text.replace("constexpr int kScoreStages = 4;", "constexpr int kScoreStages = 5;"))
    assert bench.kernel_source_hash() != base
