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



def test_point_summary_follows_the_scope_formulas():
    """The low-rank overhead is [t(K1) + t(K2)] - [t(K1, r=0) + t(K2, r=0)] over t(K2, r=0);
    %FP4 is 2MNK / t(K2) / peak; %HBM is kernel 1's algorithmic bytes / t(K1) / peak; TFLOP/s and
    tokens/s come from the forward's time.  Hand-computed on round numbers."""
    from w4a4_rank_corrected_e2m1_b300 import synthetic
    w = synthetic.scaled(synthetic.MLP_UP, M=1000, K=2000, N=3000, rank=10)
    t = {"cold": {"fwd_us": 100.0, "k1_us": 20.0, "k2_us": 90.0, "k1_rank0_us": 18.0, "k2_rank0_us": 80.0},
         "warm": {"fwd_us": 90.0, "k1_us": 15.0, "k2_us": 85.0, "k1_rank0_us": 14.0, "k2_rank0_us": 76.0}}
    s = bench.point_summary(w, t, hbm=5000.0, fp4_peak=12000.0)
    assert abs(s["lowrank_overhead"] - (110.0 - 98.0) / 80.0) < 1e-12
    assert abs(s["frac_fp4_k2"] - 2 * 1000 * 3000 * 2000 / 90e-6 / 1e12 / 12000.0) < 1e-12
    kb = 1000 * 2000 * 2 + 1000 * 2000 // 2 + 1000 * 2000 // 16 + 1000 * 10 * 2 + 2000 * 10 * 2 + 2000 * 4
    assert bench.k1_bytes(1000, 2000, 10) == kb
    assert abs(s["frac_hbm_k1"] - kb / 20e-6 / 1e9 / 5000.0) < 1e-12
    flops = 2 * 1000 * 3000 * 2000 + 2 * 1000 * 2000 * 10 + 2 * 1000 * 10 * 3000
    assert abs(s["tflops"] - flops / 100e-6 / 1e12) < 1e-9
    assert abs(s["tokens_per_s"] - 1000 / 100e-6) < 1e-6
    assert s["warm_l2"]["k2_us"] == 85.0


def test_sweep_covers_every_timed_point():
    from w4a4_rank_corrected_e2m1_b300 import synthetic
    names = [w.name for w in synthetic.SWEEP]
    assert names[0] == "flux_mlp_up" and len(names) == len(set(names)) == 10
    assert {"flux_qkv", "flux_mlp_down"} <= set(names)
    assert sorted(w.M for w in synthetic.SWEEP if w.name.startswith("flux_oproj_m")) == [256, 1024, 4096, 16384]
    assert sorted(w.rank for w in synthetic.SWEEP if w.name.startswith("flux_oproj_r")) == [16, 64, 128]
