"""CPU tests of the GPU library's host side: build, exported symbols, argument
validation, schedule geometry and the partition controller rule."""
import ctypes
import os
import re
import shutil
import subprocess
import tempfile

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


# ------------------------------------------------------------------------------------------------
# library: builds for sm_103a, loads, exports every declared symbol
# ------------------------------------------------------------------------------------------------

def declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"\b(psr_[a-z_0-9]+)\s*\(", text)
    return sorted(set(names))


def test_library_exports_every_declared_symbol(psr):
    lib = psr.load()
    names = declared_functions()
    assert len(names) >= 8
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"
    assert set(names) == set(psr.EXPORTED)
    # nothing else leaks out of the library (hidden visibility except the C ABI)
    out = subprocess.run(["nm", "-D", "--defined-only", psr.build()], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert {n for n in exported if n.startswith("psr_")} == set(names)


def test_library_is_sm103a_only(psr):
    out = subprocess.run(["cuobjdump", "--list-elf", psr.build()], capture_output=True, text=True).stdout
    assert "sm_103a" in out
    assert "sm_90" not in out and "sm_100" not in out


def test_status_strings(psr):
    assert psr.status_string(0) == "ok"
    assert "timed out" in psr.status_string(4)
    assert psr.status_string(99) == "unknown status"


def test_workspace_sizes(psr):
    import ring_inputs as ri
    for name in ("small", "h32_s32k_nc", "h32_s32k_c", "gqa_s64k_c", "long_s128k_c", "sweep_d64_P64"):
        w = ri.WORKLOADS[name]
        n = psr.workspace_bytes(psr.make_shape(w.B, w.Hq, w.Hkv, w.S, w.P, w.d, w.causal))
        slots = 2 * 2 * w.B * w.Hkv * w.S * w.d * 2  # two slots for K and for V, every (b, kvh, shard)
        assert slots <= n <= slots * 2 + (64 << 20), (name, n, slots)
    with pytest.raises(psr.PsrError):
        psr.workspace_bytes(psr.make_shape(1, 2, 2, 1000, 4, 64, False))  # L = 250: not a multiple of 256
    with pytest.raises(psr.PsrError):
        psr.workspace_bytes(psr.make_shape(1, 2, 2, 1024, 4, 96, False))  # d = 96
    with pytest.raises(psr.PsrError):
        psr.workspace_bytes(psr.make_shape(0, 2, 2, 1024, 4, 64, False))  # empty batch


def test_fwd_rejects_bad_arguments_without_touching_the_device(psr):
    lib = psr.load()
    sh = psr.make_shape(1, 2, 2, 1024, 4, 64, False)
    part = psr.make_partition()
    ok_ptr = 1 << 20
    args = [ok_ptr] * 6
    # null pointers
    for i in range(6):
        a = list(args)
        a[i] = None
        rc = lib.psr_ring_attn_fwd(ctypes.byref(sh), *a[:5], a[5], 1 << 30, ctypes.byref(part), None)
        assert rc == psr.ERR_ARG
    # misaligned workspace
    rc = lib.psr_ring_attn_fwd(ctypes.byref(sh), *args[:5], ok_ptr + 16, 1 << 30, ctypes.byref(part), None)
    assert rc == psr.ERR_ARG
    # misaligned tensor
    rc = lib.psr_ring_attn_fwd(ctypes.byref(sh), ok_ptr + 2, *args[1:5], ok_ptr, 1 << 30, ctypes.byref(part), None)
    assert rc == psr.ERR_ARG
    assert lib.psr_ring_attn_fwd(None, *args[:5], ok_ptr, 1 << 30, ctypes.byref(part), None) == psr.ERR_ARG
    st = psr.Stats()
    assert lib.psr_get_stats(None, ctypes.byref(st), None) == psr.ERR_ARG


# ------------------------------------------------------------------------------------------------
# schedule geometry (compiled from the same header the kernel uses)
# ------------------------------------------------------------------------------------------------

@pytest.fixture(scope="module")
def schedule_check():
    d = tempfile.mkdtemp(prefix="psr_sched_")
    exe = os.path.join(d, "schedule_check")
    subprocess.check_call(["g++", "-O2", "-std=c++17", os.path.join(ROOT, "tests", "schedule_check.cpp"), "-o", exe])
    return exe


SHAPES = [
    # B Hq Hkv S P d causal
    (1, 2, 2, 1024, 4, 64, 0),
    (1, 2, 2, 1024, 4, 64, 1),
    (1, 32, 32, 32768, 16, 128, 0),
    (1, 32, 32, 32768, 16, 128, 1),
    (2, 32, 8, 65536, 16, 128, 1),
    (1, 8, 8, 131072, 32, 128, 1),
    (3, 6, 2, 768, 3, 64, 1),
    (2, 4, 1, 2560, 5, 128, 0),
    (1, 1, 1, 256, 1, 64, 1),
    # causal over load-balanced shards
    (1, 2, 2, 2048, 4, 64, 2),
    (1, 32, 32, 32768, 16, 128, 2),
    (2, 32, 8, 65536, 16, 128, 2),
    (1, 8, 8, 131072, 32, 128, 2),
    (3, 6, 2, 1536, 3, 64, 2),
    (1, 1, 1, 512, 1, 64, 2),
] + [(1, 16, 16, 16384, P, d, 0) for d in (64, 128) for P in (2, 4, 8, 16, 32, 64)]


@pytest.mark.parametrize("shape", SHAPES)
def test_schedule_bounds_and_coverage(schedule_check, shape):
    out = subprocess.run([schedule_check, *map(str, shape), "113"], capture_output=True, text=True)
    assert out.returncode == 0 and out.stdout.startswith("OK"), out.stdout + out.stderr


def test_wave_cap_matches_enumeration(schedule_check):
    out = subprocess.run([schedule_check, "wave"], capture_output=True, text=True)
    assert out.returncode == 0 and out.stdout.startswith("OK"), out.stdout + out.stderr


# CTA-pair items (512 query rows): shards whose length is a multiple of 512
PAIR_SHAPES = [s for s in SHAPES if (s[3] // s[4]) % (1024 if s[6] == 2 else 512) == 0] + [
    (1, 2, 2, 2048, 2, 128, 1), (2, 8, 2, 3072, 3, 128, 1), (1, 2, 2, 2048, 2, 128, 2)]


@pytest.mark.parametrize("shape", PAIR_SHAPES)
def test_schedule_pair_items(schedule_check, shape):
    out = subprocess.run([schedule_check, *map(str, shape), "56", "2"], capture_output=True, text=True)
    assert out.returncode == 0 and out.stdout.startswith("OK"), out.stdout + out.stderr


def test_schedule_pair_rejects_short_shards(schedule_check):
    out = subprocess.run([schedule_check, "1", "16", "16", "16384", "64", "128", "0", "56", "2"], capture_output=True,
                         text=True).stdout
    assert out.startswith("REJECT")  # L = 256 cannot hold a 512-row pair item


def test_schedule_splits_large_groups(schedule_check):
    # GQA with 4 query heads per KV head and L = 4096: 64 items read one slot; a bound of 20 splits it in 4
    out = subprocess.run([schedule_check, "2", "32", "8", "65536", "16", "128", "1", "20"], capture_output=True,
                         text=True).stdout
    assert out.startswith("OK") and "Gs=16 n_sub=4" in out


SCHEDULE_MUTANTS = {
    # a chunk below the shard read in full, or its first half missed by the items
    "below_full": ("if (t <= c.r) return G.kv_tiles / 2;", "if (t < c.r) return G.kv_tiles / 2;"),
    # a chunk above the shard read only half by the second-half items
    "above_half": ("return second_half(G, c) ? G.kv_tiles : 0;", "return second_half(G, c) ? G.kv_tiles / 2 : 0;"),
    # staging copies half a chunk where the items read all of it
    "stage_half": ("return (is_balanced<kBal>(G) && t <= r) ? G.kv_tiles / 2 : G.kv_tiles;",
                   "return (is_balanced<kBal>(G) && t < r) ? G.kv_tiles / 2 : G.kv_tiles;"),
}


@pytest.mark.parametrize("name", sorted(SCHEDULE_MUTANTS))
def test_schedule_check_catches_planted_mistakes(name):
    old, new = SCHEDULE_MUTANTS[name]
    d = tempfile.mkdtemp(prefix="psr_sched_mut_")
    src = open(os.path.join(ROOT, "persistent_sm_ring_gb300", "csrc", "psr_schedule.h")).read()
    assert old in src
    os.makedirs(os.path.join(d, "persistent_sm_ring_gb300", "csrc"))
    os.makedirs(os.path.join(d, "tests"))
    with open(os.path.join(d, "persistent_sm_ring_gb300", "csrc", "psr_schedule.h"), "w") as f:
        f.write(src.replace(old, new, 1))
    shutil.copy(os.path.join(ROOT, "tests", "schedule_check.cpp"), os.path.join(d, "tests"))
    exe = os.path.join(d, "sc")
    subprocess.check_call(["g++", "-O2", "-std=c++17", os.path.join(d, "tests", "schedule_check.cpp"), "-o", exe])
    out = subprocess.run([exe, "1", "2", "2", "2048", "4", "64", "2", "113"], capture_output=True, text=True).stdout
    shutil.rmtree(d, ignore_errors=True)
    assert out.startswith("FAIL"), out


def test_schedule_balanced_rejects_half_items(schedule_check):
    # L = 256: each half of a balanced shard would hold half an item
    out = subprocess.run([schedule_check, "1", "2", "2", "1024", "4", "64", "2", "100"], capture_output=True,
                         text=True).stdout
    assert out.startswith("REJECT")


def test_library_balanced_rejects_half_items(psr):
    # L = 256: a half of a balanced shard cannot hold a whole 256-row item
    with pytest.raises(psr.PsrError):
        psr.workspace_bytes(psr.make_shape(1, 2, 2, 1024, 4, 64, psr.CAUSAL_BALANCED))
    assert psr.workspace_bytes(psr.make_shape(1, 2, 2, 2048, 4, 64, psr.CAUSAL_BALANCED)) > 0
    with pytest.raises(psr.PsrError):
        psr.workspace_bytes(psr.make_shape(1, 2, 2, 2048, 4, 64, 3))


def test_schedule_rejects_unsupported(schedule_check):
    out = subprocess.run([schedule_check, "1", "2", "2", "640", "5", "64", "0", "100"], capture_output=True,
                         text=True).stdout
    assert out.startswith("REJECT")  # L = 128 is not a multiple of 256


# ------------------------------------------------------------------------------------------------
# controller rule
# ------------------------------------------------------------------------------------------------

def test_controller_golden_values(psr):
    path = os.path.join(ROOT, "tests", "golden", "controller_rule.txt")
    n = 0
    for line in open(path):
        line = line.split("#")[0].strip()
        if not line:
            continue
        N, Rs, Cs, Rp, Cp, lo, hi, want = line.split()
        got = psr.controller_target(int(N), float(Rs), float(Cs), float(Rp), float(Cp), int(lo), int(hi))
        assert got == int(want), line
        n += 1
    assert n >= 10


def test_controller_minimises_predicted_makespan(psr):
    """The rule equalises R_s*C_s/n and R_p*C_p/(N-n); so the rounded target is
    within one block of the integer split that minimises the larger of the two
    predicted finish times (checked by exhaustive search)."""
    rng = np.random.default_rng(0)
    for _ in range(2000):
        N = int(rng.integers(2, 400))
        Rs, Rp = rng.integers(1, 10**6, size=2)
        Cs, Cp = rng.uniform(1.0, 1e5, size=2)
        n = psr.controller_target(N, Rs, Cs, Rp, Cp, 1, N)
        span = [max(Rs * Cs / k, Rp * Cp / (N - k)) for k in range(1, N)]
        best = 1 + int(np.argmin(span))
        assert abs(n - best) <= 1, (N, Rs, Cs, Rp, Cp, n, best)
        assert 1 <= n <= N - 1


# ------------------------------------------------------------------------------------------------
# GEMM workspaces: sizes and shape rules (host side only)
# ------------------------------------------------------------------------------------------------

def test_ag_gemm_workspace_holds_the_gather_buffers(psr):
    for M, K, Ns, P in [(1024, 512, 256, 4), (2048, 1024, 512, 4), (512, 256, 256, 1), (8192, 8192, 3584, 8)]:
        n = psr.ag_gemm_workspace_bytes(M, K, Ns, P)
        assert P * M * K * 2 <= n < P * M * K * 2 + (1 << 20), (M, K, Ns, P, n)  # one gathered A per rank
    for bad in [(1000, 512, 256, 4),   # M/P = 250, not a multiple of 256
                (1024, 512, 384, 4),   # Ns not a multiple of 256
                (1024, 500, 256, 4),   # K not a multiple of 128
                (1024, 512, 256, 3)]:  # M not divisible by P
        with pytest.raises(psr.PsrError):
            psr.ag_gemm_workspace_bytes(*bad)


def test_gemm_rs_workspace_holds_every_partial_tile(psr):
    # the fp32 partials of 256 x 512 output tiles: [P][M][N'] with N' = N rounded up to 512 (a
    # rank's last tile is half wide when N is an odd multiple of 256; its second half is not stored)
    for M, N, Ks, P in [(1024, 512, 256, 4), (512, 768, 192, 1), (768, 256, 320, 3), (8192, 8192, 3584, 8)]:
        n = psr.gemm_rs_workspace_bytes(M, N, Ks, P)
        part = P * M * ((N + 511) // 512 * 512) * 4
        assert part <= n < part + (1 << 20), (M, N, Ks, P, n)
    for bad in [(1024, 300, 256, 4),       # N not a multiple of 256
                (1024, 512, 100, 4),       # Ks not a multiple of 64
                (65 * 256, 512, 64, 65),   # more ranks than a reduce round holds (64)
                (1000, 512, 256, 4)]:      # M/P not a multiple of 256
        with pytest.raises(psr.PsrError):
            psr.gemm_rs_workspace_bytes(*bad)
