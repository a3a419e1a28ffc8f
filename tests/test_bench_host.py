"""Host-side logic of bench.py (no GPU): the launch count it reports and the
rule that keeps ncu traffic figures only while the kernel's sources are
unchanged."""
import json
import os
import sys
import types

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _fake_lib():
    names = ["qgemv_q4k_ex", "qgemv_q4k_group", "qgemv_q4k_fused", "qgemv_q4k_fused_group", "qgemm_q4k_batched",
             "qgemv_iq3_ex", "qgemv_iq3_group", "qgemv_iq3xxs_ex", "qgemm_iq3_batched", "qgemv_codebook",
             "qgemv_q4k_pass"]
    return types.SimpleNamespace(**{n: object() for n in names})


def test_kernel_launches_follow_the_token_groups():
    lib = _fake_lib()
    kl = bench.kernel_launches
    # Q4_K: groups of at most 4 tokens up to 4; from 5 (no prologue or
    # residual) tcgen05 per matrix and group of <= 10; batched from 16: one launch
    assert [kl(lib, lib.qgemv_q4k_ex, (), m) for m in (1, 4, 5, 8, 10, 11, 15)] == [1, 1, 1, 1, 1, 2, 2]
    assert [kl(lib, lib.qgemv_q4k_group, (None, None, None, 3), m) for m in (3, 5, 13)] == [1, 3, 6]
    assert kl(lib, lib.qgemm_q4k_batched, (), 8) == 1
    assert kl(lib, lib.qgemm_q4k_batched, (), 16) == 1
    assert kl(lib, lib.qgemv_q4k_fused_group, (), 3) == 1
    assert kl(lib, lib.qgemv_q4k_fused, (), 8) == 2
    # IQ3: groups of 4 tokens up to 4; from 5, tcgen05 per matrix and group of <= 10
    grp = (None, None, None, 3)
    assert [kl(lib, lib.qgemv_iq3_group, grp, m) for m in (1, 2, 3, 4, 5, 8, 13)] == [1, 1, 1, 1, 3, 3, 6]
    assert [kl(lib, lib.qgemv_iq3_ex, (), m) for m in (4, 5, 10, 11, 15)] == [1, 1, 1, 2, 2]
    assert kl(lib, lib.qgemm_iq3_batched, (), 8) == 1
    assert kl(lib, lib.qgemm_iq3_batched, (), 32) == 1
    assert kl(lib, lib.qgemv_iq3xxs_ex, (), 8) == 2
    # codebook formats: IQ4 (ids 1, 2) groups of 4, grid formats groups of 8
    assert kl(lib, lib.qgemv_codebook, (1,), 5) == 2
    assert kl(lib, lib.qgemv_codebook, (3,), 5) == 1
    assert kl(lib, lib.qgemv_q4k_pass, (), 1) == 1


def test_traffic_kept_only_while_sources_match(tmp_path, monkeypatch):
    entry = {"dram_bytes_per_launch": 123, "sources": "q4k",
             "kernel_source_hash": bench.kernel_source_hash(bench.KERNEL_SOURCES["q4k"])}
    stale = dict(entry, kernel_source_hash="0" * 16)
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "traffic.json").write_text(json.dumps({"a:M1": entry, "b:M1": stale}))
    csrc = os.path.join(ROOT, "block_quantised_weight_gb300", "csrc")
    (tmp_path / "block_quantised_weight_gb300").mkdir()
    os.symlink(csrc, tmp_path / "block_quantised_weight_gb300" / "csrc")
    os.symlink(os.path.join(ROOT, "include"), tmp_path / "include")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("a", 1) == 123
    assert bench.profiled_traffic("b", 1) is None
    assert bench.profiled_traffic("c", 1) is None


def test_every_kernel_source_set_exists():
    csrc = os.path.join(ROOT, "block_quantised_weight_gb300", "csrc")
    for files in bench.KERNEL_SOURCES.values():
        for f in files:
            assert os.path.exists(os.path.join(csrc, f)), f
