"""Shared-memory layouts of the GEMV kernels, checked on the host.

tests/layout_probe.cu prints, for every configuration the launchers can
choose, the layout that launch_gemv derives.  The checks are the rules the
copies into that memory depend on: mbarriers 8-byte aligned, every
tensor-map (TMA) destination and bulk-copy destination on a 128-byte
boundary, at least two ring stages inside the per-CTA limit, and each
super-block inside the box that carries it (an IQ3 block of 98 bytes starts
0..14 bytes into its 112-byte box, since the box's x coordinate is the
block's byte offset rounded down to 16).

tests/tc_layout_probe.cu does the same for the tcgen05 kernels of
gemm_tc.cu: every token count their launchers accept, with the ring rule of
launch_tc.
"""
import json
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "block_quantised_weight_gb300", "csrc")


@pytest.fixture(scope="module")
def layouts(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    exe = str(tmp_path_factory.mktemp("layout") / "layout_probe")
    subprocess.run([nvcc, "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a", "-I", CSRC,
                    "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "layout_probe.cu"), "-o", exe],
                   check=True, capture_output=True, timeout=300)
    out = subprocess.run([exe], check=True, capture_output=True, text=True, timeout=60).stdout
    return [json.loads(line) for line in out.splitlines() if line.strip()]


def test_every_configuration_is_listed(layouts):
    got = {(c["fmt"], c["MT"], c["RG"], c["MINB"], c["fuse"]) for c in layouts}
    assert ("q4k", 1, 1, 2, 0) in got and ("q4k", 4, 1, 1, 2) in got
    assert {("q4k2", 1, 1, 1, 1), ("q4k2", 1, 1, 1, 2)} <= got
    assert {("iq3", 1, 2, 1, 0), ("iq3", 2, 1, 1, 0), ("iq3", 4, 1, 1, 0)} <= got
    assert len(got) == len(layouts) == 20


def test_ring_fits_with_at_least_two_stages(layouts):
    for c in layouts:
        assert 2 <= c["stages"] <= c["max_stages"], c
        assert c["total"] <= c["budget"] <= c["smem_per_cta"], c
        assert c["total"] == c["stage0"] + c["stages"] * c["stage_bytes"], c


def test_barriers_and_copy_destinations_aligned(layouts):
    for c in layouts:
        # one full and one empty mbarrier per stage, 8 bytes each, before sx
        assert c["full"] % 8 == 0 and c["empty"] % 8 == 0, c
        assert c["empty"] >= c["full"] + 8 * c["max_stages"], c
        assert c["sx"] >= c["empty"] + 8 * c["max_stages"], c
        for k in ("sx", "red", "cred", "ss", "table", "stage0", "stage_bytes", "xoff", "aoff"):
            assert c[k] % 128 == 0, (k, c)
        # weight boxes: one per block column at st + b * tile_rows * box_bytes
        assert (c["tile_rows"] * c["box_bytes"]) % 128 == 0, c
        assert c["xoff"] >= c["cols"] * c["tile_rows"] * c["box_bytes"], c
        # x: per token a padded 2D box (IQ3) or one 1 KB-per-column bulk copy (Q4_K)
        x_per_token = c["x_box_bytes"] if c["xh"] == 132 else c["cols"] * 1024
        assert x_per_token % 128 == 0, c
        assert c["aoff"] - c["xoff"] >= c["MT"] * x_per_token, c
        # prologue operands: the RMSNorm weight once, the SwiGLU up operand per token
        extra = {0: 0, 1: c["cols"] * 1024, 2: c["MT"] * c["cols"] * 1024}[c["fuse"]]
        assert c["stage_bytes"] - c["aoff"] == extra, c


def test_per_warp_arrays_hold_every_consumer_warp(layouts):
    """Each consumer warp owns MT x 8 sub-block sums of x, two tile
    parities of MT x 32 row sums and two of MT sums of x^2: with two warps
    per column (q4k2) there are 16 warps, not 8."""
    for c in layouts:
        w, mt = c["warps"], c["MT"]
        assert c["red"] - c["sx"] >= w * mt * 8 * 4, c
        assert c["cred"] - c["red"] >= 2 * w * mt * 32 * 4, c
        assert c["table"] - c["ss"] >= 2 * w * mt * 4, c


def test_tables_sit_between_reductions_and_ring(layouts):
    for c in layouts:
        iq3 = c["fmt"].startswith("iq3")
        assert c["stage0"] - c["table"] == (256 * 32 * 8 + 128 * 16 * 8 if iq3 else 0), c
        assert c["table"] >= c["ss"], c


def test_every_block_lies_inside_its_box(layouts):
    for c in layouts:
        for col in range(64):  # the block's offset modulo 16 repeats every 8 columns
            start = col * c["block_bytes"]
            box_x = start & ~15  # the tensor-map x coordinate: a multiple of 16 bytes
            assert box_x % 16 == 0
            assert start - box_x + c["block_bytes"] <= c["box_bytes"], (c["fmt"], col)


@pytest.fixture(scope="module")
def tc_layouts(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    exe = str(tmp_path_factory.mktemp("tc_layout") / "tc_layout_probe")
    subprocess.run([nvcc, "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a", "-I", CSRC,
                    "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "tc_layout_probe.cu"), "-o", exe],
                   check=True, capture_output=True, timeout=300)
    out = subprocess.run([exe], check=True, capture_output=True, text=True, timeout=60).stdout
    return [json.loads(line) for line in out.splitlines() if line.strip()]


def test_tc_every_token_count_is_listed(tc_layouts):
    got = {(c["fmt"], c["xp"], c["M"]) for c in tc_layouts}
    assert got == ({(0, 1, m) for m in range(16, 33)} | {(1, 1, m) for m in range(16, 33)}
                   | {(1, 3, m) for m in range(1, 11)} | {(2, 3, m) for m in range(1, 11)})


def test_tc_rings_fit_and_align(tc_layouts):
    """At least two raw stages within the per-CTA limit; the raw ring, each
    stage and its x part (a TMA destination) on 1024-byte boundaries; the x
    stages (swizzled MMA operands) on 1024-byte boundaries; nothing below the
    ring reaches into it; the W box inside the stage's W part."""
    for c in tc_layouts:
        assert 2 <= c["nraw"] and c["smem"] <= c["smem_max"], c
        assert c["raw0"] % 1024 == 0 and c["stage"] % 1024 == 0 and c["raw_w"] % 1024 == 0, c
        assert c["below"] <= c["raw0"], c
        assert c["b0"] % 1024 == 0 and c["b_stage"] % 1024 == 0 and c["b0"] + 4 * c["b_stage"] <= c["below"], c
        assert c["box_bytes"] * c["tile_rows"] <= c["raw_w"], c


def test_tc_operands_and_tensor_memory(tc_layouts):
    """x rows (token parts) fit a 32-row atom and the MMA's N; the mbarriers
    end below the TMEM address slot; every TMEM column used is allocated."""
    for c in tc_layouts:
        assert c["x_rows"] <= 32 and c["x_rows"] <= c["ncol"] and c["ncol"] in (16, 32), c
        assert c["barrier_bytes"] <= c["tmem_slot"], c
        assert c["tmem_end"] <= c["tmem_cols"] == 512, c
