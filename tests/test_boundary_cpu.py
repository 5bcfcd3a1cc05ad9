"""Host-only tests of the C-ABI library: it loads without a GPU, exports every
function include/tpgemm.h declares, rejects bad arguments with the documented
status before anything is launched, and its tile scheduler partitions the
output exactly (each tile owned by one CTA: "cuTile Rust explained",
"Ownership crosses the launch boundary")."""
import ctypes
import os
import re
import subprocess

import pytest

import tile_partitioned_dense_gb300 as tpd
from tile_partitioned_dense_gb300 import build_ext

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tpgemm.h")


@pytest.fixture(scope="module", autouse=True)
def built():
    build_ext.build()
    tpd.load_library()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gemm_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ["gemm_create", "gemm_run", "gemm_destroy", "gemm_sync_status", "gemm_status_string"]:
        assert required in names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(tpd.LIB_PATH)
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    out = subprocess.run(["nm", "-D", "--defined-only", tpd.LIB_PATH], capture_output=True, text=True)
    if out.returncode == 0:
        exported = set(re.findall(r"\sT\s(\w+)", out.stdout))
        for n in _declared_functions():
            assert n in exported, n


def test_status_strings():
    for code, name in [(0, "TPGEMM_OK"), (-1, "TPGEMM_ERR_INVALID_ARG"), (-2, "TPGEMM_ERR_ALIGNMENT"),
                       (-3, "TPGEMM_ERR_OVERLAP"), (-4, "TPGEMM_ERR_UNSUPPORTED_DEVICE"),
                       (-5, "TPGEMM_ERR_CUDA"), (-6, "TPGEMM_ERR_TIMEOUT"), (-7, "TPGEMM_ERR_TOO_LARGE")]:
        assert tpd.gemm_status_string(code) == name
    assert tpd.gemm_status_string(123) == "TPGEMM_ERR_UNKNOWN"


def test_null_handle_is_rejected_without_gpu():
    assert tpd.gemm_run(None, 8, 8, 8, 0x1000, 8, 0x2000, 8, None, 8, 0x3000, 8, 1.0, 0.0, 0, None) == tpd.ERR_INVALID_ARG
    assert tpd.gemm_sync_status(None, None) == tpd.ERR_INVALID_ARG
    assert tpd.gemm_destroy(None) == tpd.OK
    assert tpd.gemm_force_variant(None, 0) == tpd.ERR_INVALID_ARG
    assert tpd.gemm_watchdog_selftest(None, 10000, None) == tpd.ERR_INVALID_ARG
    assert tpd.gemm_num_sms(None) == tpd.ERR_INVALID_ARG
    assert tpd.gemm_set_workspace(None, 0x1000, 1 << 24, None) == tpd.ERR_INVALID_ARG
    assert tpd.gemm_workspace_size(None) == tpd.ERR_INVALID_ARG
    assert tpd.gemm_plan_tail_ksplit(None, 4096, 4096, 4096, tpd.OUT_BF16) == tpd.ERR_INVALID_ARG


# Fake, well-separated, 16-byte aligned device addresses: gemm_check_args only
# compares and aligns pointers.
A0, B0, C0, D0 = 0x10000000, 0x20000000, 0x30000000, 0x40000000


def chk(M=64, N=64, K=64, A=A0, lda=None, B=B0, ldb=None, C=None, ldc=None, D=D0, ldd=None, beta=0.0,
        out=tpd.OUT_BF16):
    lda = K if lda is None else lda
    ldb = N if ldb is None else ldb
    ldc = N if ldc is None else ldc
    ldd = N if ldd is None else ldd
    return tpd.gemm_check_args(M, N, K, A, lda, B, ldb, C, ldc, D, ldd, beta, out)


def test_check_args_accepts_valid():
    assert chk() == tpd.OK
    assert chk(C=C0, beta=1.0) == tpd.OK
    assert chk(M=4096, N=4096, K=4096) == tpd.OK
    assert chk(out=tpd.OUT_F32, C=C0, beta=-2.0) == tpd.OK
    assert chk(M=1, K=7, lda=7) == tpd.OK  # one row: its stride is never used


def test_check_args_invalid():
    assert chk(out=2) == tpd.ERR_INVALID_ARG
    assert chk(M=-1) == tpd.ERR_INVALID_ARG
    assert chk(K=-3) == tpd.ERR_INVALID_ARG
    assert chk(D=None) == tpd.ERR_INVALID_ARG
    assert chk(A=None) == tpd.ERR_INVALID_ARG
    assert chk(B=None) == tpd.ERR_INVALID_ARG
    assert chk(beta=1.0, C=None) == tpd.ERR_INVALID_ARG
    assert chk(lda=56) == tpd.ERR_INVALID_ARG
    assert chk(ldb=56) == tpd.ERR_INVALID_ARG
    assert chk(ldd=56) == tpd.ERR_INVALID_ARG
    assert chk(C=C0, ldc=56, beta=1.0) == tpd.ERR_INVALID_ARG


def test_check_args_too_large():
    assert chk(M=2 ** 31) == tpd.ERR_TOO_LARGE
    assert chk(K=2 ** 31, lda=2 ** 31) == tpd.ERR_TOO_LARGE


def test_check_args_alignment():
    assert chk(A=A0 + 8) == tpd.ERR_ALIGNMENT
    assert chk(B=B0 + 2) == tpd.ERR_ALIGNMENT
    assert chk(D=D0 + 4) == tpd.ERR_ALIGNMENT
    assert chk(C=C0 + 8, beta=1.0) == tpd.ERR_ALIGNMENT
    assert chk(K=60, lda=60) == tpd.ERR_ALIGNMENT    # 120-byte rows
    assert chk(N=60, ldb=60, ldd=64) == tpd.ERR_ALIGNMENT
    assert chk(N=60, ldb=64, ldd=60) == tpd.ERR_ALIGNMENT
    assert chk(N=60, ldb=64, ldd=60, out=tpd.OUT_F32) == tpd.OK  # 240 bytes is a 16-byte multiple
    assert chk(K=60, lda=64) == tpd.OK


def test_check_args_overlap():
    # D inside A
    assert chk(D=A0 + 64 * 16) == tpd.ERR_OVERLAP
    # D overlapping B's last row
    assert chk(D=B0 + 63 * 64 * 2) == tpd.ERR_OVERLAP
    # in place D == C, same stride: allowed
    assert chk(C=D0, beta=1.0) == tpd.OK
    # D == C with a different stride, or a shifted C: rejected
    assert chk(C=D0, ldc=72, beta=1.0) == tpd.ERR_OVERLAP
    assert chk(C=D0 + 16, beta=1.0) == tpd.ERR_OVERLAP
    # C may alias D freely when it is not read (beta == 0)
    assert chk(C=D0 + 16, beta=0.0) == tpd.OK
    # A and B may overlap each other (both read-only)
    assert chk(B=A0) == tpd.OK
    # adjacent, not overlapping
    assert chk(D=A0 + 64 * 64 * 2) == tpd.OK


def test_check_args_degenerate():
    assert chk(M=0, A=None, B=None, D=None) == tpd.OK
    assert chk(N=0, A=None, B=None, D=None) == tpd.OK
    assert chk(K=0, A=None, B=None) == tpd.OK
    assert chk(K=0, A=None, B=None, C=C0, beta=2.0) == tpd.OK


def test_create_without_gpu_fails_cleanly():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p()
    st = tpd.load_library().gemm_create(ctypes.byref(h), 0)
    assert st in (tpd.ERR_CUDA, tpd.ERR_INVALID_ARG)
    assert not h.value


def _tile_grid(M, N, bm=128, bn=256):
    return (M + bm - 1) // bm, (N + bn - 1) // bn


GRIDS = [_tile_grid(256, 256), _tile_grid(4096, 4096), _tile_grid(8192, 6144), _tile_grid(8192, 4096),
         _tile_grid(4096, 4096, bm=256), _tile_grid(8192, 6144, bm=256), _tile_grid(8192, 4096, bm=256),
         (1, 1), (3, 7), (17, 5), (64, 1), (1, 224), (20, 8), (10, 8)]


@pytest.mark.parametrize("mt,nt", GRIDS)
@pytest.mark.parametrize("cap", [1, 7, 74, 76, 148, 152, 160, 1000])
@pytest.mark.parametrize("group_m", [1, 8, 16])
@pytest.mark.parametrize("mode", ["whole", "cta", "pair"])
def test_schedule_is_an_exact_partition(mt, nt, cap, group_m, mode):
    """Every 64-column granule of every tile row is owned by exactly one worker."""
    pair, split = mode == "pair", mode != "whole"
    workers = tpd.gemm_schedule_workers(mt, nt, cap, pair, split)
    assert 1 <= workers <= cap
    owner = {}
    loads = []
    narrowest = 256 if not split else (128 if pair else 64)
    for w in range(workers):
        items = tpd.gemm_schedule_tiles(mt, nt, group_m, cap, w, pair, split)
        load = 0
        for (m, n0, width) in items:
            assert 0 <= m < mt and 0 <= n0 and n0 + width <= nt * 256
            assert width in (256, 128, 64) and width >= narrowest and n0 % width == 0
            for c in range(n0 // 64, (n0 + width) // 64):
                assert (m, c) not in owner, f"columns {c * 64}.. of tile row {m} owned twice"
                owner[(m, c)] = w
            load += width
        loads.append(load)
    assert tpd.gemm_schedule_tiles(mt, nt, group_m, cap, workers, pair, split) == []  # past the last worker
    assert len(owner) == mt * nt * 4
    # balance: no worker does more than one whole tile beyond another
    assert max(loads) - min(loads) <= 256


def test_schedule_tail_split_balances_square():
    # square 4096^3 in pair mode: 16 x 16 tiles of 256 x 256 on 76 pairs = 3 whole
    # rounds + 28 tiles, which are cut into 56 halves: nobody does a 4th whole tile.
    loads = [sum(x[2] for x in tpd.gemm_schedule_tiles(16, 16, 8, 76, w, True)) for w in range(76)]
    assert max(loads) == 3 * 256 + 128 and min(loads) == 3 * 256
    # without splitting the busiest workers own four whole tiles
    loads = [sum(x[2] for x in tpd.gemm_schedule_tiles(16, 16, 8, 76, w, True, False)) for w in range(76)]
    assert max(loads) == 4 * 256


def test_schedule_split_choice_follows_the_cost_model():
    # A piece 1/f wide costs a + (1 - a)/f of a tile (a = 1/3 for 1-CTA tiles).
    # 160 tiles on 152 CTAs: 8 left over -> quarters (one round at 1/2 a tile)
    assert tpd.gemm_schedule_tiles(20, 8, 16, 152, 0)[-1][2] == 64
    # 222 tiles: 70 left -> halves (1 round at 2/3) beat quarters (2 rounds at 1/2)
    assert tpd.gemm_schedule_tiles(222, 1, 16, 152, 0)[-1][2] == 128
    # 252 tiles: 100 left -> halves would take 2 rounds at 2/3 > 1 whole round
    assert all(x[2] == 256 for x in tpd.gemm_schedule_tiles(252, 1, 16, 152, 0))
    # a 128-row chunk of an 8192-wide output: 32 tiles on 152 CTAs -> 128 quarter tiles
    assert tpd.gemm_schedule_workers(1, 32, 152) == 128
    items = [tpd.gemm_schedule_tiles(1, 32, 16, 152, w) for w in range(128)]
    assert all(len(i) == 1 and i[0][2] == 64 for i in items)
    # pairs (halves at most, a = 1/2): 32 pair tiles on 76 pairs -> 64 halves
    assert tpd.gemm_schedule_workers(1, 32, 76, True) == 64


# Co-resident clusters of 2, 3 and 4 CTAs of the streaming kernel that the
# occupancy API reported on a 152-SM GB300 (any ring depth).
GB300_CLUSTERS = (76, 46, 36)


@pytest.mark.parametrize("nt,kb,mt,want", [
    (224, 64, 16, 2),   # decode 16x28672x4096: 3 rounds of 76 pairs (1.53) beat 2 rounds of 152 CTAs (2.0)
    (48, 64, 16, 2),    # N = 6144: one round of 48 pairs (0.51); 46 triples would need a second round (0.69)
    (40, 64, 32, 3),    # N = 5120: one round of triples (0.35) beats pairs (0.51) and quads (2 rounds, 0.53)
    (32, 224, 16, 4),   # 16x4096x14336: one round of 32 quads (0.27)
    (112, 64, 16, 1),   # N = 14336: one round of 112 CTAs (1.0) beats 2 rounds of pairs (1.02)
    (32, 1, 16, 1),     # a single K block cannot be split
    (32, 2, 16, 2),     # two K blocks: at most two parts
    (4, 128, 64, 3),    # 64 token rows: four parts leave too small a ring, so three
])
def test_stream_split_choice(nt, kb, mt, want):
    assert tpd.gemm_stream_split(nt, kb, mt, 152, GB300_CLUSTERS) == want


def test_stream_split_skips_impossible_cluster_sizes():
    # no cluster of 3 or 4 fits: 40 panels fall back to pairs
    assert tpd.gemm_stream_split(40, 64, 16, 152, (76, 0, 0)) == 2
    # nothing but single CTAs
    assert tpd.gemm_stream_split(40, 64, 16, 152, (0, 0, 0)) == 1
    lib = tpd.load_library()
    arr = (ctypes.c_int32 * 3)(76, 46, 36)
    for bad in [(0, 64, 16, 152), (40, 0, 16, 152), (40, 64, 8, 152), (40, 64, 80, 152), (40, 64, 24, 152),
                (40, 64, 16, 0)]:
        assert lib.gemm_stream_split(*bad, arr) == tpd.ERR_INVALID_ARG, bad
    assert lib.gemm_stream_split(40, 64, 16, 152, None) == tpd.ERR_INVALID_ARG


@pytest.mark.parametrize("tiles,kb,want", [
    (32, 64, 4),    # 256 x 4096 x 4096: 32 tiles, each on a cluster of four
    (36, 64, 4),    # as many tiles as clusters of four
    (37, 64, 2),    # one more: clusters of two
    (64, 64, 2),    # 512 x 4096: 64 tiles on 64 pairs of CTAs
    (76, 64, 2),
    (77, 64, 1),    # more tiles than pairs: the persistent schedule
    (224, 64, 1),   # 256 x 28672: plenty of tiles
    (8, 3, 2),      # three K blocks: at most two parts
    (8, 1, 1),      # a single K block cannot be shared
])
def test_tiled_ksplit_choice(tiles, kb, want):
    assert tpd.gemm_tiled_ksplit(tiles, kb, 76, 36) == want


def test_tiled_ksplit_rejects_bad_arguments():
    lib = tpd.load_library()
    for bad in [(0, 64, 76, 36), (8, 0, 76, 36), (8, 64, -1, 36), (8, 64, 76, -1)]:
        assert lib.gemm_tiled_ksplit(*bad) == tpd.ERR_INVALID_ARG, bad
    # no cluster of either size fits: no split
    assert tpd.gemm_tiled_ksplit(8, 64, 0, 0) == 1


def test_schedule_grouped_raster_order():
    # the first tiles of a band walk down the band before moving right
    order = tpd.gemm_schedule_tiles(40, 8, 16, 1, 0)
    assert [(m, n) for (m, n, _) in order[:16]] == [(m, 0) for m in range(16)]
    assert [(m, n) for (m, n, _) in order[16:20]] == [(m, 256) for m in range(4)]
    # the last band has 40 - 32 = 8 rows
    tail = order[32 * 8:32 * 8 + 9]
    assert [(m, n) for (m, n, _) in tail[:8]] == [(32 + m, 0) for m in range(8)] and tail[8][:2] == (32, 256)


def test_schedule_rejects_bad_arguments():
    lib = tpd.load_library()
    assert lib.gemm_schedule_tiles(4, 4, 0, 1, 0, 1, 0, None, 0) == tpd.ERR_INVALID_ARG
    assert lib.gemm_schedule_tiles(4, 4, 8, 2, 0, 1, -1, None, 0) == tpd.ERR_INVALID_ARG
    assert lib.gemm_schedule_tiles(4, 4, 8, 2, 0, 1, 0, None, 3) == tpd.ERR_INVALID_ARG
    assert lib.gemm_schedule_workers(4, 4, 0, 0, 1) == tpd.ERR_INVALID_ARG


# The K split tail's rule for CTA-pair schedules (gemm_run applies the same
# function): column halves only, at least 32 K blocks, and a workspace that
# holds 4 KB of flags plus four 64 KB partial-sum slots per left-over tile.
def test_tail_workspace_bytes():
    assert tpd.gemm_tail_workspace_bytes(0) == 4096
    assert tpd.gemm_tail_workspace_bytes(28) == 4096 + 28 * 4 * 65536
    assert tpd.gemm_tail_workspace_bytes(-1) == tpd.ERR_INVALID_ARG


@pytest.mark.parametrize("split,kb,tiles,ws_mult,want", [
    (2, 64, 28, 1, 1),    # square 4096^3: 28 left over, 64 K blocks
    (2, 32, 28, 1, 1),    # the threshold itself
    (2, 31, 28, 1, 0),    # one K block short: the exchange would not pay
    (1, 64, 28, 1, 0),    # no halves (mlp_down: 56 left over on 76 pairs)
    (2, 64, 28, 0, 0),    # workspace one byte too small
    (2, 64, 0, 1, 0),     # no partial round
])
def test_tail_ksplit_choice(split, kb, tiles, ws_mult, want):
    ws = tpd.gemm_tail_workspace_bytes(tiles) - (0 if ws_mult else 1)
    assert tpd.gemm_tail_ksplit(split, kb, tiles, ws) == want


def test_tail_ksplit_rejects_bad_arguments():
    for bad in [(0, 64, 1, 1 << 24), (2, 0, 1, 1 << 24), (2, 64, -1, 1 << 24), (2, 64, 1, -1)]:
        assert tpd.gemm_tail_ksplit(*bad) == tpd.ERR_INVALID_ARG, bad


# ---------------------------------------------------------------- block-scaled (MX) argument checks

def mx_chk(M=128, N=128, K=256, A=A0, lda=None, fa=0, SA=0x50000000, B=B0, ldb=None, fb=0, SB=0x60000000, C=None,
           ldc=None, D=D0, ldd=None, beta=0.0, out=tpd.OUT_BF16):
    lda = K if lda is None else lda
    ldb = K if ldb is None else ldb
    ldc = N if ldc is None else ldc
    ldd = N if ldd is None else ldd
    return tpd.gemm_mx_check_args(M, N, K, A, lda, fa, SA, B, ldb, fb, SB, C, ldc, D, ldd, beta, out)


def test_mx_scale_bytes():
    assert tpd.gemm_mx_scale_bytes(128, 128) == 512
    assert tpd.gemm_mx_scale_bytes(129, 128) == 1024
    assert tpd.gemm_mx_scale_bytes(128, 160) == 1024
    assert tpd.gemm_mx_scale_bytes(8192, 4096) == 64 * 32 * 512
    assert tpd.gemm_mx_scale_bytes(0, 4096) == 0
    assert tpd.gemm_mx_scale_bytes(-1, 32) == tpd.ERR_INVALID_ARG


def test_mx_check_args():
    assert mx_chk() == tpd.OK
    assert mx_chk(K=96) == tpd.OK
    assert mx_chk(K=100) == tpd.ERR_INVALID_ARG
    assert mx_chk(fa=2) == tpd.ERR_INVALID_ARG and mx_chk(fb=-1) == tpd.ERR_INVALID_ARG
    assert mx_chk(out=5) == tpd.ERR_INVALID_ARG
    assert mx_chk(lda=128) == tpd.ERR_INVALID_ARG and mx_chk(ldb=255) == tpd.ERR_INVALID_ARG
    assert mx_chk(lda=264) == tpd.ERR_ALIGNMENT and mx_chk(ldb=264) == tpd.ERR_ALIGNMENT
    assert mx_chk(M=1, lda=264) == tpd.OK  # one row: its stride is not used
    assert mx_chk(SA=0x50000008) == tpd.ERR_ALIGNMENT and mx_chk(SB=0x60000004) == tpd.ERR_ALIGNMENT
    assert mx_chk(SA=None) == tpd.ERR_INVALID_ARG
    assert mx_chk(M=2 ** 31) == tpd.ERR_TOO_LARGE
    assert mx_chk(M=0) == tpd.OK and mx_chk(N=0, D=None) == tpd.OK
    assert mx_chk(K=0, A=None, B=None, SA=None, SB=None) == tpd.OK
    assert mx_chk(beta=1.0) == tpd.ERR_INVALID_ARG  # C missing
    assert mx_chk(beta=1.0, C=D0) == tpd.OK          # in place
    assert mx_chk(beta=1.0, C=D0 + 16) == tpd.ERR_OVERLAP
    assert mx_chk(D=0x50000000 + 256) == tpd.ERR_OVERLAP  # D inside A's scales
    assert mx_chk(D=A0 + 64) == tpd.ERR_OVERLAP
    assert mx_chk(D=B0) == tpd.ERR_OVERLAP


def test_mx_null_handle():
    assert tpd.gemm_run_mx(None, 8, 8, 32, A0, 32, 0, 0x50000000, B0, 32, 0, 0x60000000, None, 8, D0, 8, 1.0, 0.0,
                           tpd.OUT_F32, None) == tpd.ERR_INVALID_ARG


# ---------------------------------------------------------------- block-scaled FP4 argument checks

def fp4_chk(M=128, N=128, K=256, fmt=tpd.NVFP4, A=A0, lda=None, SA=0x50000000, B=B0, ldb=None, SB=0x60000000,
            C=None, ldc=None, D=D0, ldd=None, beta=0.0, out=tpd.OUT_BF16):
    lda = K // 2 if lda is None else lda
    ldb = K // 2 if ldb is None else ldb
    ldc = N if ldc is None else ldc
    ldd = N if ldd is None else ldd
    return tpd.gemm_fp4_check_args(M, N, K, fmt, A, lda, SA, B, ldb, SB, C, ldc, D, ldd, beta, out)


def test_fp4_scale_bytes():
    nv, mx = tpd.NVFP4, tpd.MXFP4
    # NVFP4: a chunk per 128 rows and 64 elements of K; MXFP4: per 128 elements
    assert tpd.gemm_fp4_scale_bytes(nv, 128, 64) == 512
    assert tpd.gemm_fp4_scale_bytes(nv, 128, 80) == 1024
    assert tpd.gemm_fp4_scale_bytes(nv, 129, 64) == 1024
    assert tpd.gemm_fp4_scale_bytes(nv, 8192, 4096) == 64 * 64 * 512
    assert tpd.gemm_fp4_scale_bytes(mx, 8192, 4096) == tpd.gemm_mx_scale_bytes(8192, 4096)
    assert tpd.gemm_fp4_scale_bytes(mx, 128, 160) == 1024
    assert tpd.gemm_fp4_scale_bytes(nv, 0, 4096) == 0
    assert tpd.gemm_fp4_scale_bytes(nv, -1, 16) == tpd.ERR_INVALID_ARG
    assert tpd.gemm_fp4_scale_bytes(2, 128, 64) == tpd.ERR_INVALID_ARG


def test_fp4_check_args():
    assert fp4_chk() == tpd.OK and fp4_chk(fmt=tpd.MXFP4) == tpd.OK
    assert fp4_chk(K=96) == tpd.OK and fp4_chk(K=96, fmt=tpd.MXFP4) == tpd.OK
    assert fp4_chk(K=80, lda=48, ldb=48) == tpd.OK                            # 16-element blocks
    assert fp4_chk(K=80, lda=48, ldb=48, fmt=tpd.MXFP4) == tpd.ERR_INVALID_ARG  # not whole 32-element blocks
    assert fp4_chk(K=100) == tpd.ERR_INVALID_ARG
    assert fp4_chk(fmt=2) == tpd.ERR_INVALID_ARG and fp4_chk(fmt=-1) == tpd.ERR_INVALID_ARG
    assert fp4_chk(out=5) == tpd.ERR_INVALID_ARG
    assert fp4_chk(lda=64) == tpd.ERR_INVALID_ARG and fp4_chk(ldb=127) == tpd.ERR_INVALID_ARG  # < K/2 bytes
    assert fp4_chk(lda=136) == tpd.ERR_ALIGNMENT and fp4_chk(ldb=136) == tpd.ERR_ALIGNMENT
    assert fp4_chk(M=1, lda=136) == tpd.OK  # one row: its stride is not used
    assert fp4_chk(SA=0x50000008) == tpd.ERR_ALIGNMENT and fp4_chk(SB=0x60000004) == tpd.ERR_ALIGNMENT
    assert fp4_chk(SA=None) == tpd.ERR_INVALID_ARG
    assert fp4_chk(M=2 ** 31) == tpd.ERR_TOO_LARGE
    assert fp4_chk(M=0) == tpd.OK and fp4_chk(N=0, D=None) == tpd.OK
    assert fp4_chk(K=0, A=None, B=None, SA=None, SB=None) == tpd.OK
    assert fp4_chk(beta=1.0) == tpd.ERR_INVALID_ARG  # C missing
    assert fp4_chk(beta=1.0, C=D0) == tpd.OK          # in place
    assert fp4_chk(beta=1.0, C=D0 + 16) == tpd.ERR_OVERLAP
    assert fp4_chk(D=0x50000000 + 1024) == tpd.ERR_OVERLAP  # D inside A's scales (2 KB for NVFP4 here)
    assert fp4_chk(D=0x50000000 + 1024, fmt=tpd.MXFP4) == tpd.OK  # past MXFP4's 1 KB
    assert fp4_chk(D=A0 + 64) == tpd.ERR_OVERLAP
    assert fp4_chk(D=B0) == tpd.ERR_OVERLAP


def test_fp4_null_handle():
    assert tpd.gemm_run_fp4(None, 8, 8, 64, tpd.NVFP4, A0, 32, 0x50000000, B0, 32, 0x60000000, None, 8, D0, 8, 1.0,
                            0.0, tpd.OUT_F32, None) == tpd.ERR_INVALID_ARG
