"""bench.py ties each committed ncu record to the kernel sources it was taken
on through kernel_source_hash: the hash must survive comment-only and
layout-only edits and change with any edit to the code itself."""
import os
import shutil

import bench


def _copy_tree(tmp_path):
    root = tmp_path / "repo"
    pkg = root / "quantized_kv_cache_03_gb300"
    (pkg / "csrc").mkdir(parents=True)
    (root / "include").mkdir()
    src_pkg = os.path.join(bench.ROOT, "quantized_kv_cache_03_gb300")
    for k in bench.KERNEL_SOURCES.values():
        for f in k:
            shutil.copy(os.path.join(src_pkg, f), pkg / f)
    shutil.copy(os.path.join(bench.ROOT, "include", "kvq.h"), root / "include" / "kvq.h")
    return root


def test_hash_ignores_comments_and_layout_but_not_code(tmp_path, monkeypatch):
    root = _copy_tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(root))
    h0 = {k: bench.kernel_source_hash(k) for k in bench.KERNEL_SOURCES}
    f = root / "quantized_kv_cache_03_gb300" / "csrc" / "kvq_prefill.cuh"
    text = f.read_text()
    # comment lines added and removed, a block comment, re-indentation
    edited = "// a new comment line\n// and another\n" + text.replace("namespace kvq {", "namespace kvq {   /* note */\n\n", 1)
    edited = edited.replace("    ", "  ")
    f.write_text(edited)
    assert {k: bench.kernel_source_hash(k) for k in bench.KERNEL_SOURCES} == h0
    # a one-character code edit changes the prefill hash (and only that one)
    f.write_text(edited.replace("constexpr float kSlack = 3.0f;", "constexpr float kSlack = 4.0f;", 1))
    h1 = {k: bench.kernel_source_hash(k) for k in bench.KERNEL_SOURCES}
    assert h1["prefill_attn"] != h0["prefill_attn"] and h1["split_attn"] == h0["split_attn"]
    # the shared header feeds both
    g = root / "quantized_kv_cache_03_gb300" / "csrc" / "kvq_internal.cuh"
    g.write_text(g.read_text().replace("namespace kvq {", "namespace kvq { constexpr int kProbe = 1;", 1))
    h2 = {k: bench.kernel_source_hash(k) for k in bench.KERNEL_SOURCES}
    assert h2["split_attn"] != h0["split_attn"] and h2["prefill_attn"] != h1["prefill_attn"]
