"""bench.source_sha keys the committed ncu records: it must follow the CUDA
sources' code and ignore their comments."""
import os

import bench


def _tree(tmp_path, text):
    csrc = tmp_path / "bidirectional_selective_scan_vssm_b300" / "csrc"
    csrc.mkdir(parents=True, exist_ok=True)
    (csrc / "k.cuh").write_text(text)
    (csrc / "notes.txt").write_text("not a source file")
    return str(tmp_path)


def test_source_sha_ignores_comments_not_code(tmp_path, monkeypatch):
    code = "int f(int a)\n{\n    return a + 1;\n}\n"
    monkeypatch.setattr(bench, "ROOT", _tree(tmp_path, code))
    base = bench.source_sha()
    commented = ("// header\n/* block\n comment */\nint f(int a)   // trailing\n{\n\n"
                 "    return a + 1;  /* inline */\n}\n")
    monkeypatch.setattr(bench, "ROOT", _tree(tmp_path, commented))
    assert bench.source_sha() == base
    monkeypatch.setattr(bench, "ROOT", _tree(tmp_path, code.replace("a + 1", "a + 2")))
    assert bench.source_sha() != base


def test_source_sha_of_the_tree_is_stable():
    assert bench.source_sha() == bench.source_sha()
    assert len(bench.source_sha()) == 16
    assert os.path.isdir(os.path.join(bench.ROOT, "bidirectional_selective_scan_vssm_b300", "csrc"))
