"""Host-side pieces of bench.py that need no GPU."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_traffic_read_from_a_matching_profile_only(tmp_path, monkeypatch):
    import hashlib
    csrc = tmp_path / "sparse_paged_kv_page_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    src = csrc / "k.cu"
    src.write_text("// kernel\n")
    sha = hashlib.sha256(src.read_bytes()).hexdigest()
    (tmp_path / "profiles" / "k.md").write_text(
        "# k\n\n```\nncu --set full -k regex:\"a|b\" -o x\n```\n\n"
        f"- source_sha256: `{sha}` (k.cu when captured)\n"
        "- dram_bytes_per_launch_full_size: 205709056\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_from_profile("k.cu", "k.md") == 205709056.0
    src.write_text("// kernel, changed\n")             # the summary no longer applies
    assert bench.traffic_from_profile("k.cu", "k.md") is None
    assert bench.traffic_from_profile("k.cu", "missing.md") is None


def test_byte_models():
    from sa_synth import config
    c = config(5)
    # 3 statistics rows of D bf16 per (page, KV head)
    assert bench.score_bytes(c, [16 * 10]) == 10 * c.H_kv * 3 * c.D * 2
    assert bench.score_bytes(c, [16 * 10 + 1]) == 11 * c.H_kv * 3 * c.D * 2


def test_entmax_byte_model_reads_v_only_for_kept_rows():
    from sa_synth import config
    c = config(5)
    L = 16 * 1000
    full = bench.step_bytes(c, [L])
    # every selected token kept: the softmax step's bytes
    all_rows = c.topk * c.ps * c.H_kv
    assert bench.entmax_step_bytes(c, [L], all_rows) == full
    # no V row read: K of the selection, the statistics, q and out
    assert full - bench.entmax_step_bytes(c, [L], 0) == all_rows * c.D * 2
