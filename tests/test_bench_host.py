"""Host-side bookkeeping of bench.py (no GPU): the key that ties recorded DRAM traffic to a
kernel's code."""
import bench


def _hash_of(tmp_path, monkeypatch, text):
    d = tmp_path / "w4a4_rank_corrected_e2m1_b300" / "csrc"
    d.mkdir(parents=True, exist_ok=True)
    (d / "k.cu").write_text(text)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "KERNEL_SOURCES", {"k": ["k.cu"]})
    return bench.kernel_source_hash("k")


CODE = "__global__ void k(int* p) {\n  p[0] = 1;\n}\n"


def test_comment_and_whitespace_edits_keep_the_key(tmp_path, monkeypatch):
    base = _hash_of(tmp_path, monkeypatch, CODE)
    commented = "// a note\n/* a block\n   comment */\n__global__ void k(int* p) {   // store\n\n  p[0] = 1;\n}\n"
    assert _hash_of(tmp_path, monkeypatch, commented) == base


def test_code_edits_change_the_key(tmp_path, monkeypatch):
    base = _hash_of(tmp_path, monkeypatch, CODE)
    assert _hash_of(tmp_path, monkeypatch, CODE.replace("p[0] = 1", "p[0] = 2")) != base

