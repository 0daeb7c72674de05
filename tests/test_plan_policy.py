"""The plan's launch policy (csrc/mfr_policy.h) on the CPU: which kernel,
how many CTAs per token, threads and grid for a call of T tokens of width H.

The header is pure host C++; this test compiles it into a small shared
library with the host compiler and checks the choices the design notes
state, the edges of every threshold, the even spread of the persistent
grid, and the refusals."""
import ctypes
import os
import subprocess

import numpy as np
import pytest

import moe_finalize_residual_rmsnorm_gb300 as mfr

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(ROOT, "moe_finalize_residual_rmsnorm_gb300", "csrc")
INCLUDE = os.path.join(ROOT, "include")
SMS = 152
RING_THREADS = 544
ERR_ARG, ERR_SHAPE = 1, 2      # MFR_ERR_INVALID_ARG, MFR_ERR_UNSUPPORTED_SHAPE

SHIM = r'''
#include "mfr_policy.h"
extern "C" int policy_choose(long long T, long long H, int k, int fused, int fp4, int en, int fv, int cs,
                             int stages, int sms, int* out, char* err, int errn) {
    mfr::PolicyIn in{T, H, k, fused != 0, fp4 != 0, en != 0, fv, cs, stages, sms};
    mfr::PolicyOut o{};
    const int rc = mfr::choose_launch(in, &o, err, static_cast<size_t>(errn), 544);
    out[0] = o.variant; out[1] = o.cluster; out[2] = o.cpt; out[3] = o.block; out[4] = o.grid_x;
    out[5] = o.early_trigger;
    return rc;
}
extern "C" int policy_stream_grid(long long T, int sms) { return mfr::stream_grid(T, sms); }
extern "C" int policy_all_slots(long long T, long long H, int k, int fused, int fp4, int en) {
    return mfr::ring_all_slots(T, H, k, fused != 0, fp4 != 0, en != 0) ? 1 : 0;
}
'''


@pytest.fixture(scope="module")
def lib(tmp_path_factory):
    d = tmp_path_factory.mktemp("policy")
    src = d / "shim.cpp"
    src.write_text(SHIM)
    so = d / "libpolicy.so"
    subprocess.run(["g++", "-O1", "-std=c++17", "-shared", "-fPIC", f"-I{CSRC}", f"-I{INCLUDE}", str(src),
                    "-o", str(so)], check=True)
    L = ctypes.CDLL(str(so))
    L.policy_choose.restype = ctypes.c_int
    L.policy_choose.argtypes = [ctypes.c_longlong, ctypes.c_longlong] + [ctypes.c_int] * 8 + \
        [ctypes.POINTER(ctypes.c_int), ctypes.c_char_p, ctypes.c_int]
    L.policy_stream_grid.restype = ctypes.c_int
    L.policy_stream_grid.argtypes = [ctypes.c_longlong, ctypes.c_int]
    L.policy_all_slots.restype = ctypes.c_int
    L.policy_all_slots.argtypes = [ctypes.c_longlong, ctypes.c_longlong] + [ctypes.c_int] * 4
    return L


def choose(lib, T, H, k=8, fused=True, fp4=False, en=False, variant=mfr.VARIANT_AUTO, cluster=0, stages=5):
    out = (ctypes.c_int * 6)()
    err = ctypes.create_string_buffer(200)
    rc = lib.policy_choose(T, H, k, int(fused), int(fp4), int(en), variant, cluster, stages, SMS, out, err, 200)
    keys = ("variant", "cluster", "cpt", "block", "grid_x", "early_trigger")
    return rc, dict(zip(keys, list(out))), err.value.decode()


AUTO_TABLE = [
    # (T, H, variant, CTAs per token)
    (1, 4096, mfr.VARIANT_CLUSTER, 4), (4, 4096, mfr.VARIANT_CLUSTER, 4), (5, 4096, mfr.VARIANT_CLUSTER, 16),
    (8, 4096, mfr.VARIANT_CLUSTER, 16), (32, 4096, mfr.VARIANT_CLUSTER, 16), (33, 4096, mfr.VARIANT_CLUSTER, 8),
    (64, 4096, mfr.VARIANT_CLUSTER, 8), (65, 4096, mfr.VARIANT_CLUSTER, 2), (128, 4096, mfr.VARIANT_CLUSTER, 2),
    (129, 4096, mfr.VARIANT_ROWS, 1), (304, 4096, mfr.VARIANT_ROWS, 1), (305, 4096, mfr.VARIANT_STREAM, 1),
    (384, 4096, mfr.VARIANT_STREAM, 1),
    (16384, 4096, mfr.VARIANT_STREAM, 1),
    (1, 8192, mfr.VARIANT_CLUSTER, 8), (2, 8192, mfr.VARIANT_CLUSTER, 8), (3, 8192, mfr.VARIANT_CLUSTER, 16),
    (16, 8192, mfr.VARIANT_CLUSTER, 16), (32, 8192, mfr.VARIANT_CLUSTER, 8), (64, 8192, mfr.VARIANT_CLUSTER, 4),
    (65, 8192, mfr.VARIANT_ROWS, 1), (152, 8192, mfr.VARIANT_ROWS, 1), (153, 8192, mfr.VARIANT_STREAM, 1),
    (192, 8192, mfr.VARIANT_STREAM, 1),
    (2, 1024, mfr.VARIANT_ROWS, 1), (32, 1024, mfr.VARIANT_CLUSTER, 4), (1, 16384, mfr.VARIANT_CLUSTER, 16),
]


@pytest.mark.parametrize("T,H,variant,cluster", AUTO_TABLE)
def test_automatic_choice(lib, T, H, variant, cluster):
    rc, o, _ = choose(lib, T, H)
    assert rc == mfr.MFR_OK
    assert (o["variant"], o["cluster"]) == (variant, cluster)
    if variant == mfr.VARIANT_STREAM:
        assert o["block"] == RING_THREADS and o["early_trigger"] == 0
    else:
        assert o["grid_x"] == T * cluster
        assert o["early_trigger"] == (1 if T * H <= 1 << 19 else 0)
        chunks = H // 8 // cluster
        assert o["cpt"] * o["block"] >= chunks and o["block"] % 32 == 0 and o["block"] <= 512


PLAIN_TABLE = [(1, 4096, 8), (2, 4096, 8), (4, 4096, 16), (8, 4096, 2), (16, 4096, 2), (32, 4096, 4),
               (128, 4096, 4), (1, 8192, 16), (2, 8192, 16), (4, 8192, 4), (8, 8192, 4), (16, 8192, 8),
               (64, 8192, 8)]


@pytest.mark.parametrize("T,H,cluster", PLAIN_TABLE)
def test_plain_finalize_split(lib, T, H, cluster):
    """The plain finalize splits a token's columns over CTAs that share
    nothing; its split sizes are its own."""
    rc, o, _ = choose(lib, T, H, fused=False)
    assert rc == 0 and (o["variant"], o["cluster"]) == (mfr.VARIANT_CLUSTER, cluster)
    assert o["block"] * o["cpt"] * cluster >= H // 8


def test_one_cta_geometry(lib):
    for H, cpt, block in ((24, 1, 32), (4096, 1, 512), (4104, 2, 288), (8192, 2, 512), (16384, 4, 512)):
        rc, o, _ = choose(lib, 300, H, variant=mfr.VARIANT_ROWS)
        assert rc == 0 and (o["cpt"], o["block"], o["grid_x"]) == (cpt, block, 300), H


def test_persistent_grid_spreads_tokens_evenly(lib):
    for T in range(1, 5001):
        g = lib.policy_stream_grid(T, SMS)
        rounds = -(-T // SMS)
        assert 1 <= g <= SMS
        assert -(-T // g) == rounds                      # no extra round
        loads = [len(range(b, T, g)) for b in range(g)]
        assert max(loads) - min(loads) <= 1              # every CTA within one token of the others
        assert g == T or g == -(-T // rounds)            # as few CTAs as that allows


def test_forced_variants_and_cluster_sizes(lib):
    rc, o, _ = choose(lib, 16, 4096, variant=mfr.VARIANT_CLUSTER, cluster=2)
    assert rc == 0 and (o["variant"], o["cluster"], o["block"]) == (mfr.VARIANT_CLUSTER, 2, 256)
    rc, o, _ = choose(lib, 16, 4096, variant=mfr.VARIANT_CLUSTER)            # auto size when forced
    assert rc == 0 and o["cluster"] == 8
    rc, o, _ = choose(lib, 16, 32, variant=mfr.VARIANT_CLUSTER)              # narrow: still split in 2
    assert rc == 0 and (o["variant"], o["cluster"], o["block"]) == (mfr.VARIANT_CLUSTER, 2, 32)
    for H in (24, 4104):                                                      # 3 and 513 chunks
        rc, o, err = choose(lib, 16, H, variant=mfr.VARIANT_CLUSTER, cluster=2)
        assert rc == ERR_SHAPE and "divisible" in err
    rc, o, _ = choose(lib, 5, 4096, variant=mfr.VARIANT_STREAM)
    assert rc == 0 and o["variant"] == mfr.VARIANT_STREAM and o["grid_x"] == 5
    rc, _, err = choose(lib, 500, 4096, variant=mfr.VARIANT_STREAM, stages=1)
    assert rc == ERR_SHAPE and "stages" in err
    rc, o, _ = choose(lib, 5000, 4096, stages=1)                              # no ring room: one CTA per token
    assert rc == 0 and o["variant"] == mfr.VARIANT_ROWS


def test_nvfp4_rules(lib):
    rc, _, err = choose(lib, 4, 4104, fp4=True)
    assert rc == ERR_SHAPE and "16" in err
    # blocks of 16 columns never straddle two CTAs: 514 chunks split in 2 gives 257, odd
    rc, o, _ = choose(lib, 4, 4112, fp4=True, variant=mfr.VARIANT_CLUSTER, cluster=2)
    assert rc == 0 and o["variant"] == mfr.VARIANT_ROWS and o["cluster"] == 1
    rc, o, _ = choose(lib, 1, 4096, fp4=True)
    assert rc == 0 and o["cluster"] == 4
    for T, H, cluster in ((8, 4096, 16), (32, 4096, 8), (16, 8192, 16), (64, 4096, 8)):
        rc, o, _ = choose(lib, T, H, fp4=True)                               # 64-thread CTAs at 2^17
        assert rc == 0 and o["cluster"] == cluster, (T, H, o)


def test_per_expert_rmsnorm_rules(lib):
    ok = dict(fused=False, en=True, stages=7)
    rc, o, _ = choose(lib, 16384, 4096, **ok)
    assert rc == 0 and o["variant"] == mfr.VARIANT_STREAM
    rc, o, _ = choose(lib, 256, 4096, **ok)
    assert rc == 0 and (o["variant"], o["cluster"]) == (mfr.VARIANT_ROWS, 1)
    for T, H, cluster in ((1, 4096, 4), (2, 4096, 4), (4, 4096, 16), (8, 4096, 16), (16, 4096, 8),
                          (32, 4096, 1), (128, 4096, 1), (1, 8192, 8), (2, 8192, 16), (4, 8192, 16),
                          (8, 8192, 16), (16, 8192, 2), (32, 8192, 2), (64, 8192, 1)):
        rc, o, _ = choose(lib, T, H, **ok)
        want = mfr.VARIANT_CLUSTER if cluster > 1 else mfr.VARIANT_ROWS
        assert rc == 0 and (o["variant"], o["cluster"]) == (want, cluster), (T, H, o)
    rc, o, _ = choose(lib, 1, 4096, k=16, fused=False, en=True, stages=3)
    assert rc == 0 and (o["variant"], o["cluster"]) == (mfr.VARIANT_ROWS, 1)  # more than 8 slots
    rc, o, _ = choose(lib, 16384, 4096, k=16, fused=False, en=True, stages=3)
    assert rc == 0 and o["variant"] == mfr.VARIANT_ROWS                      # more than 8 slots
    rc, _, _ = choose(lib, 16384, 4096, k=16, fused=False, en=True, stages=3, variant=mfr.VARIANT_STREAM)
    assert rc == ERR_SHAPE
    rc, _, _ = choose(lib, 64, 16384, fused=False, en=True, stages=7, variant=mfr.VARIANT_STREAM)
    assert rc == ERR_SHAPE                                                     # more than 4 tiles
    rc, o, _ = choose(lib, 16384, 8192, fused=False, en=True, stages=2, variant=mfr.VARIANT_STREAM)
    assert rc == 0 and o["variant"] == mfr.VARIANT_STREAM                    # two stages are enough
    rc, o, _ = choose(lib, 16384, 8192, fused=False, en=True, stages=1)
    assert rc == 0 and o["variant"] == mfr.VARIANT_ROWS
    rc, _, _ = choose(lib, 16384, 8192, fused=False, en=True, stages=1, variant=mfr.VARIANT_STREAM)
    assert rc == ERR_SHAPE
    rc, o, _ = choose(lib, 64, 4096, fused=False, en=True, stages=7, variant=mfr.VARIANT_CLUSTER)
    assert rc == 0 and o["variant"] == mfr.VARIANT_CLUSTER and o["cluster"] == 8
    rc, _, _ = choose(lib, 64, 4096, k=9, fused=False, en=True, stages=7, variant=mfr.VARIANT_CLUSTER)
    assert rc == ERR_SHAPE


def test_every_choice_fits_its_kernel(lib):
    """Over many shapes, plan kinds and options, whatever the policy returns
    is a geometry its kernel can run: whole warps, at most 512 threads, every
    16-byte chunk owned by one thread, a cluster that splits the chunks
    evenly (NVFP4: whole 16-column blocks per CTA), the per-expert cluster
    and one-pass forms within 8 slots, the ring within its slot and tile
    limits, and the persistent grid no larger than the SM count."""
    rng = np.random.default_rng(123)
    variants = (mfr.VARIANT_AUTO, mfr.VARIANT_CLUSTER, mfr.VARIANT_ROWS, mfr.VARIANT_STREAM)
    checked = 0
    for _ in range(20000):
        H = int(rng.integers(1, 2049)) * 8
        T = int(rng.choice([1, 2, 3, 5, 8, 16, 33, 64, 100, 128, 200, 512, 1000, 4096, 20000]))
        k = int(rng.integers(1, 17))
        kind = int(rng.integers(0, 4))          # 0 fused, 1 plain, 2 NVFP4, 3 per-expert
        fused, fp4, en = kind in (0, 2), kind == 2, kind == 3
        if fp4 and H % 16:
            continue
        variant = int(rng.choice(variants))
        cluster = int(rng.choice([0, 0, 1, 2, 4, 8, 16]))
        stages = int(rng.integers(0, 9))
        rc, o, err = choose(lib, T, H, k=k, fused=fused, fp4=fp4, en=en, variant=variant, cluster=cluster,
                            stages=stages)
        if rc != mfr.MFR_OK:
            assert rc in (ERR_ARG, ERR_SHAPE) and err, (T, H, k, kind, variant, cluster, stages)
            continue
        checked += 1
        chunks = H // 8
        assert o["variant"] in (mfr.VARIANT_CLUSTER, mfr.VARIANT_ROWS, mfr.VARIANT_STREAM)
        if variant != mfr.VARIANT_AUTO:
            assert o["variant"] == variant or (variant == mfr.VARIANT_CLUSTER and o["variant"] == mfr.VARIANT_ROWS)
        if o["variant"] == mfr.VARIANT_STREAM:
            assert stages >= 2 and o["block"] == RING_THREADS and 1 <= o["grid_x"] <= min(T, SMS)
            assert -(-H // 2048) <= 8
            if en:
                assert k <= 8 and H <= 8192
            continue
        c = o["cluster"]
        assert c in (1, 2, 4, 8, 16) and chunks % c == 0
        assert (c > 1) == (o["variant"] == mfr.VARIANT_CLUSTER)
        per_cta = chunks // c
        assert o["cpt"] in (1, 2, 4) and o["block"] % 32 == 0 and 32 <= o["block"] <= 512
        assert o["block"] * o["cpt"] >= per_cta and (o["block"] - 32) * o["cpt"] < per_cta
        assert o["grid_x"] == T * c
        if fp4 and c > 1:
            assert per_cta % 2 == 0
        if en and c > 1:
            assert k <= 8 and o["cpt"] <= 2
    assert checked > 5000


def test_ring_all_slots_instantiation(lib):
    """The ring kernel takes the no-per-slot-test instantiation for k = 8:
    the residual + bf16 form up to 2^24 elements at H <= 8192, the plain
    finalize at every size up to H = 4096 and up to 2^22 elements at
    H = 8192; never for other k, the NVFP4 output or wider rows."""
    a = lambda T, H, k=8, fused=1, fp4=0, en=0: lib.policy_all_slots(T, H, k, fused, fp4, en)
    assert a(1, 4096) == 1 and a(4096, 4096) == 1 and a(4097, 4096) == 0 and a(16384, 4096) == 0
    assert a(2048, 8192) == 1 and a(2049, 8192) == 0 and a(32768, 8192) == 0
    assert a(2730, 6144) == 1 and a(2731, 6144) == 0
    assert a(16000, 1032) == 1
    assert a(100, 8200) == 0 and a(100, 16384) == 0
    fin = lambda T, H, k=8: a(T, H, k=k, fused=0)
    assert fin(16384, 4096) == 1 and fin(1 << 20, 2048) == 1
    assert fin(512, 8192) == 1 and fin(513, 8192) == 0 and fin(8192, 8192) == 0
    assert fin(100, 8200) == 0 and fin(100, 16384) == 0
    for k in (1, 4, 7, 9, 16):
        assert a(1000, 4096, k=k) == 0 and fin(1000, 4096, k=k) == 0
    assert a(1000, 4096, fp4=1) == 0 and a(1000, 4096, fused=0, en=1) == 0


def test_rows_to_ring_at_one_wave(lib):
    """One CTA per token while its grid is one wave (8192 elements per SM:
    304 tokens at H = 4096, 152 at H = 8192), the ring above, for the
    residual + bf16, plain finalize and per-expert RMSNorm outputs; the
    NVFP4 output keeps one CTA per token below 1.5 * 2^20 elements."""
    for kw in (dict(), dict(fused=False), dict(fused=False, en=True)):
        for T, H, want in ((304, 4096, mfr.VARIANT_ROWS), (305, 4096, mfr.VARIANT_STREAM),
                           (152, 8192, mfr.VARIANT_ROWS), (153, 8192, mfr.VARIANT_STREAM)):
            rc, o, _ = choose(lib, T, H, **kw)
            assert rc == 0 and o["variant"] == want, (kw, T, H)
    for T, H, want in ((305, 4096, mfr.VARIANT_ROWS), (383, 4096, mfr.VARIANT_ROWS), (384, 4096, mfr.VARIANT_STREAM),
                       (191, 8192, mfr.VARIANT_ROWS), (192, 8192, mfr.VARIANT_STREAM)):
        rc, o, _ = choose(lib, T, H, fp4=True)
        assert rc == 0 and o["variant"] == want, (T, H)
