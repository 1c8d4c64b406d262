"""CPU test of the kernels' work decomposition (zigzag units, CP-step key walk).

Compiles tests/schedule_check.cpp against the kernels' schedule header with
the host compiler and checks, by brute force, that every allowed (query, key)
pair is computed exactly once.
"""
import os
import random
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))

GEOMS = [
    # b, s, hq, hkv, cp, causal, grid
    (1, 256, 2, 2, 1, 1, 3),
    (1, 512, 4, 4, 2, 1, 148),
    (2, 1024, 4, 2, 2, 1, 5),
    (1, 960, 6, 2, 3, 1, 7),
    (1, 640, 3, 1, 2, 1, 4),
    (1, 1536, 8, 1, 4, 1, 152),
    (1, 96, 2, 2, 3, 1, 2),
    (1, 2048, 2, 2, 8, 1, 11),
    (1, 768, 4, 4, 3, 0, 6),
    (2, 384, 2, 1, 1, 0, 3),
    (1, 1280, 2, 1, 5, 1, 9),
    # degenerate chunks: one token per half-chunk (s = 2cp), and two
    (1, 2, 1, 1, 1, 1, 1),
    (3, 8, 2, 1, 4, 1, 5),
    (1, 6, 3, 3, 3, 0, 2),
    (2, 16, 4, 2, 4, 1, 3),
    # odd head groups with an even number of tiles per chunk: the forward pairs
    # two query tiles of one head (MHA, G = 3, no mask, ragged second tile)
    (1, 2048, 4, 4, 4, 1, 7),
    (2, 1024, 3, 3, 2, 1, 9),
    (1, 1024, 3, 1, 2, 0, 5),
    (1, 4096, 2, 2, 2, 1, 13),
    (1, 960, 6, 2, 3, 1, 7),
    (1, 1920, 2, 2, 3, 1, 5),     # three tiles per chunk: head pairs
]


@pytest.fixture(scope="module")
def checker(tmp_path_factory):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    exe = str(tmp_path_factory.mktemp("sched") / "schedule_check")
    subprocess.run([cxx, "-O2", "-std=c++17", "-o", exe, os.path.join(HERE, "schedule_check.cpp")], check=True)
    return exe


def test_fast_division_matches_integer_division(checker):
    """The unit decodes divide by multiply and shift (FastDiv): exact against
    plain integer division for every divisor up to 5000 around each multiple,
    at the top of the range, and for two million random pairs."""
    out = subprocess.run([checker, "D"], capture_output=True, text=True)
    assert out.returncode == 0 and out.stdout.strip() == "ok fastdiv", out.stdout


# tile pairs in unit blocks (b, s, hq, hkv, cp, causal, grid, KV pairs per block): the
# blocks the library forms for large K/V, forced here on small shapes -- MHA, G = 3,
# no mask, a ragged second tile
BLOCKED = [
    (2, 2048, 8, 8, 4, 1, 7, 3),
    (2, 1024, 9, 3, 2, 1, 5, 1),
    (1, 1024, 5, 5, 2, 0, 3, 2),
    (3, 800, 4, 4, 2, 1, 5, 2),
    (4, 4096, 4, 4, 4, 1, 19, 2),
]


def test_tile_pair_unit_blocks_cover_every_pair_once(checker):
    """Blocks change only the order of the forward's units: every allowed pair is
    still computed once (whole sequence and rank-local form), each block longest
    first, and the padded slots decode to empty units."""
    args = []
    for *g, kv in BLOCKED:
        args += ["K", str(kv), "U", *map(str, g), "R", *map(str, g)]
    out = subprocess.run([checker, *args], capture_output=True, text=True)
    assert out.returncode == 0 and "FAIL" not in out.stdout, out.stdout
    lines = out.stdout.strip().splitlines()
    assert len(lines) == 2 * len(BLOCKED) and all(ln.startswith("ok ") for ln in lines)
    # every whole-sequence geometry forms blocks; a rank's share has fewer
    # units per head, so some of them stay one block
    assert all("[blocks of" in ln for ln in lines if "rank-local" not in ln), out.stdout
    assert sum("[blocks of" in ln for ln in lines if "rank-local" in ln) >= 2, out.stdout


# packed samples: lengths (each divisible by 2cp, 0 allowed), hq, hkv, cp, causal, grid
PACKED = [
    ([512, 256, 1024], 4, 2, 2, 1, 7),
    ([960, 0, 192, 384], 6, 2, 3, 1, 5),
    ([2048, 128], 8, 1, 4, 1, 152),
    ([96], 2, 2, 3, 1, 2),
    ([768, 1536], 2, 2, 3, 0, 4),
    ([16, 16, 16, 16, 16, 16], 3, 1, 1, 1, 3),
    ([4, 8, 0, 4], 2, 1, 2, 1, 3),                  # one- and two-token chunks
]


def test_every_allowed_pair_once(checker):
    args = [str(x) for g in GEOMS for x in ("U", *g)]
    out = subprocess.run([checker, *args], capture_output=True, text=True)
    assert out.returncode == 0, out.stdout + out.stderr
    assert out.stdout.count("ok") == len(GEOMS)


def test_packed_samples_never_cross_a_boundary(checker):
    args = []
    for lens, hq, hkv, cp, causal, grid in PACKED:
        args += ["P", str(len(lens)), *map(str, lens), str(hq), str(hkv), str(cp), str(causal), str(grid)]
    out = subprocess.run([checker, *args], capture_output=True, text=True)
    assert out.returncode == 0, out.stdout + out.stderr
    assert out.stdout.count("ok") == len(PACKED)


def _fuzz_geometries(n, seed):
    """Seeded random geometries: batch 1-3, cp 1-6, chunk 1-300 tokens, GQA
    groups 1-4, either mask, grids from 1 to 160 CTAs (sizes kept small for
    the checker's per-pair table)."""
    rng = random.Random(seed)
    out = []
    while len(out) < n:
        b, cp, c = rng.randint(1, 3), rng.randint(1, 6), rng.randint(1, 300)
        s = 2 * cp * c
        hkv = rng.randint(1, 2)
        hq = hkv * rng.randint(1, 4)
        if b * s > 2400:
            continue
        out.append((b, s, hq, hkv, cp, rng.randint(0, 1), rng.randint(1, 160)))
    return out


def test_random_geometries(checker):
    geoms = _fuzz_geometries(24, seed=2026)
    args = [str(x) for g in geoms for x in ("U", *g)]
    out = subprocess.run([checker, *args], capture_output=True, text=True)
    assert out.returncode == 0, out.stdout + out.stderr
    assert out.stdout.count("ok") == len(geoms)


def test_random_packed_geometries(checker):
    rng = random.Random(7)
    args, n = [], 0
    while n < 12:
        cp = rng.randint(1, 4)
        lens = [2 * cp * rng.randint(0, 60) for _ in range(rng.randint(1, 6))]
        if sum(lens) == 0 or sum(lens) > 2000:
            continue
        hkv = rng.randint(1, 2)
        hq = hkv * rng.randint(1, 3)
        args += ["P", str(len(lens)), *map(str, lens), str(hq), str(hkv), str(cp), str(rng.randint(0, 1)),
                 str(rng.randint(1, 40))]
        n += 1
    out = subprocess.run([checker, *args], capture_output=True, text=True)
    assert out.returncode == 0, out.stdout + out.stderr
    assert out.stdout.count("ok") == n


def test_rank_local_form_covers_every_pair_once(checker):
    """One rank's share of a CP group over GPUs (the all-gather form, the ring
    form step by step, and the backward over every key tile): over all ranks,
    with local rows mapped back to the sequence, every allowed pair once and
    every addressed row inside its buffer. Fixed geometries plus seeded random
    ones."""
    geoms = [g for g in GEOMS if g[4] <= 4] + _fuzz_geometries(16, seed=4242)
    args = [str(x) for g in geoms for x in ("R", *g)]
    out = subprocess.run([checker, *args], capture_output=True, text=True)
    assert out.returncode == 0, out.stdout + out.stderr
    assert out.stdout.count("ok") == len(geoms)
