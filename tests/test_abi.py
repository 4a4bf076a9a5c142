"""C ABI checks that need no GPU: the library builds for sm_103a, loads, and
exports every function include/*.h declares; argument validation; the
host-side selector."""
import ctypes
import glob
import os
import re

import pytest

import rmsnorm_fwd_gb300 as rn
from rmsnorm_fwd_gb300 import inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SMS = 152
OPTIN = 232448  # opt-in shared memory per block on sm_100-class parts (227 KiB)


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        for m in re.finditer(r"\b([a-z_][a-z0-9_]*)\s*\(", src):
            name = m.group(1)
            # a declaration: preceded by a return type on the same statement
            if name.startswith("rmsnorm_"):
                names.add(name)
    return names


def test_library_exports_every_declared_symbol():
    lib = rn._load()
    names = declared_functions()
    assert {"rmsnorm_create", "rmsnorm_fwd", "rmsnorm_destroy"} <= names
    for name in sorted(names):
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"
    # exported with C linkage (no mangling): dlsym by the plain name worked above
    assert rn.rmsnorm_version() >> 16 == 1


def test_library_is_in_tree():
    path = rn.library_path()
    assert os.path.commonpath([path, ROOT]) == ROOT
    assert os.path.exists(path)


def test_status_strings():
    for code in range(10):
        s = rn.rmsnorm_status_string(code)
        assert s and s != "unknown status"
    assert rn.rmsnorm_status_string(999) == "unknown status"


# ------------------------------------------------------------- validation (no GPU touched)

FAKE = 1 << 40  # never dereferenced: every case below fails validation first


def call(x, w, y, rows, hidden, eps, dtype):
    return rn._load().rmsnorm_fwd(x, w, y, rows, hidden, eps, dtype, None)


def test_bad_dtype():
    assert call(FAKE, FAKE + 2 ** 30, FAKE + 2 ** 31, 4, 64, 1e-6, 7) == rn.ERR_UNSUPPORTED_DTYPE


@pytest.mark.parametrize("rows,hidden,eps", [(-1, 64, 1e-6), (4, 0, 1e-6), (4, -3, 1e-6),
                                             (4, 64, -1e-6), (4, 64, float("nan")),
                                             (4, 64, float("inf"))])
def test_bad_shape_or_eps(rows, hidden, eps):
    assert call(FAKE, FAKE + 2 ** 30, FAKE + 2 ** 31, rows, hidden, eps, rn.BF16) == \
        rn.ERR_INVALID_ARG


def test_null_pointers():
    assert call(0, FAKE, FAKE + 2 ** 31, 4, 64, 1e-6, rn.BF16) == rn.ERR_INVALID_ARG
    assert call(FAKE, 0, FAKE + 2 ** 31, 4, 64, 1e-6, rn.BF16) == rn.ERR_INVALID_ARG
    assert call(FAKE, FAKE + 2 ** 30, 0, 4, 64, 1e-6, rn.BF16) == rn.ERR_INVALID_ARG


def test_partial_overlap_rejected():
    # y starts one row into x: partial overlap
    assert call(FAKE, FAKE + 2 ** 30, FAKE + 128, 4, 64, 1e-6, rn.BF16) == rn.ERR_ALIASING
    # y overlaps the weight
    assert call(FAKE, FAKE + 2 ** 30, FAKE + 2 ** 30 - 64, 4, 64, 1e-6, rn.BF16) == \
        rn.ERR_ALIASING


def test_no_context_without_gpu():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    # valid arguments: the context lookup fails (no device) before any launch
    rc = call(FAKE, FAKE + 2 ** 30, FAKE + 2 ** 31, 4, 64, 1e-6, rn.BF16)
    assert rc in (rn.ERR_CUDA, rn.ERR_NOT_INITIALIZED)
    assert rn._load().rmsnorm_create() in (rn.ERR_CUDA, rn.ERR_UNSUPPORTED_DEVICE)


# ------------------------------------------------------------- selector (host only)

A = 1 << 30  # 1 GiB-aligned fake addresses


def plan(rows, hidden, dtype, variant=rn.VARIANT_AUTO, xoff=0, sms=SMS):
    return rn.rmsnorm_plan_status(A + xoff, 3 * A, 5 * A + xoff, rows, hidden, dtype, sms,
                                  OPTIN, variant)


def test_selector_on_the_workloads():
    expect = {
        "f32_64x128": rn.VARIANT_WARP_PER_ROW,  # 512 B rows, decode-sized row count
        "embed_bf16_8192x1024": rn.VARIANT_WARP_PER_ROW,
        "prefill_bf16_16384x4096": rn.VARIANT_CTA_PER_ROW,
        "decode_bf16_1x4096": rn.VARIANT_PERSISTENT,
        "decode_bf16_8x4096": rn.VARIANT_PERSISTENT,
        "decode_bf16_32x4096": rn.VARIANT_PERSISTENT,
    }
    for name, wl in inputs.WORKLOADS.items():
        rc, p = plan(wl.rows, wl.hidden, rn.DTYPE_CODES[wl.dtype])
        assert rc == rn.OK, name
        assert p.variant != rn.VARIANT_GENERIC, name
        if name in expect:
            assert p.variant == expect[name], (name, p.as_dict())
        assert p.grid >= 1 and p.block_threads % 32 == 0 and p.block_threads <= 1024


def test_decode_one_block_per_row():
    for rows in (1, 8, 32):
        rc, p = plan(rows, 4096, rn.BF16)
        assert rc == rn.OK and p.variant == rn.VARIANT_PERSISTENT
        assert p.grid == rows
        assert p.vecs_per_thread * p.threads_per_row * 8 >= 4096


def test_persistent_grid_capped_by_sms():
    rc, p = plan(100000, 4096, rn.BF16, rn.VARIANT_PERSISTENT)
    assert rc == rn.OK and p.grid <= SMS * (2048 // p.block_threads)


def test_capacity_covers_row():
    for dt, es in ((rn.F32, 4), (rn.BF16, 2), (rn.F16, 2)):
        for hidden in (8, 64, 128, 1000, 1024, 2880, 4096, 5120, 7168, 8192, 16384, 32768):
            if hidden * es % 16:
                continue
            for v in (rn.VARIANT_WARP_PER_ROW, rn.VARIANT_CTA_PER_ROW, rn.VARIANT_PERSISTENT):
                rc, p = plan(4096, hidden, dt, v)
                if rc == rn.OK and p.vecs_per_thread > 0:  # 0: looped, any length
                    cap = p.threads_per_row * p.vecs_per_thread * p.vec_bytes // es
                    assert cap >= hidden, (dt, hidden, v, p.as_dict())


def test_ragged_rows_go_generic():
    for hidden in (1, 3, 7, 9, 31, 33, 127, 129, 1023, 1025, 8191):
        rc, p = plan(64, hidden, rn.BF16)
        assert rc == rn.OK and p.variant == rn.VARIANT_GENERIC, hidden


def test_misaligned_pointer_goes_generic_or_is_refused_when_forced():
    rc, p = plan(64, 4096, rn.BF16, xoff=2)
    assert rc == rn.OK and p.variant == rn.VARIANT_GENERIC
    for v in (rn.VARIANT_WARP_PER_ROW, rn.VARIANT_CTA_PER_ROW, rn.VARIANT_STAGED):
        rc, _ = plan(64, 4096, rn.BF16, v, xoff=2)
        assert rc == rn.ERR_MISALIGNED


def test_forced_variant_that_cannot_fit():
    rc, _ = plan(64, 16384, rn.BF16, rn.VARIANT_WARP_PER_ROW)  # 2048 vectors > 32 x 16
    assert rc == rn.ERR_VARIANT
    rc, _ = plan(64, 1 << 20, rn.BF16, rn.VARIANT_STAGED)  # 2 MiB row > shared memory
    assert rc == rn.ERR_VARIANT


def test_staged_plan_fits_and_is_consistent():
    for hidden in (2880, 4096, 5120, 7168, 16384, 32768):
        for dt in (rn.BF16, rn.F16, rn.F32):
            rc, p = plan(65536, hidden, dt, rn.VARIANT_STAGED)
            es = 4 if dt == rn.F32 else 2
            if hidden * es * 3 + 1024 > OPTIN:
                assert rc == rn.ERR_VARIANT
                continue
            assert rc == rn.OK, (hidden, dt)
            consumers = p.block_threads // 32 - 1
            wpr = p.threads_per_row // 32
            assert consumers % wpr == 0
            assert p.stages % (consumers // wpr) == 0 and p.stages >= 2
            assert p.smem_bytes <= OPTIN
            assert p.grid <= SMS


def test_prefill_rules():
    """The automatic plan for prefill shapes: lane groups for short rows,
    lean blocks of <= 256 threads with 2-4 vectors each up to 16 KiB rows,
    a persistent grid beyond."""
    for hidden, variant in ((64, rn.VARIANT_WARP_PER_ROW), (512, rn.VARIANT_WARP_PER_ROW),
                            (768, rn.VARIANT_WARP_PER_ROW), (1024, rn.VARIANT_WARP_PER_ROW),
                            (1536, rn.VARIANT_PERSISTENT), (4096, rn.VARIANT_CTA_PER_ROW),
                            (8192, rn.VARIANT_CTA_PER_ROW), (16384, rn.VARIANT_PERSISTENT),
                            (24576, rn.VARIANT_STAGED), (32768, rn.VARIANT_STAGED),
                            (65536, rn.VARIANT_CTA_PER_ROW)):
        rc, p = plan(100000, hidden, rn.BF16)
        assert rc == rn.OK and p.variant == variant, (hidden, p.as_dict())
        if variant == rn.VARIANT_CTA_PER_ROW and hidden <= 8192:
            assert p.block_threads <= 256 and 2 <= p.vecs_per_thread <= 4
        if variant == rn.VARIANT_STAGED:
            assert p.stages >= 2 and p.threads_per_row >= 128
    rc, p = plan(16384, 4096, rn.BF16)
    assert (p.block_threads, p.vecs_per_thread, p.grid) == (256, 2, 16384)
    # the same row bytes give the same shape for f32
    rc2, p2 = plan(16384, 2048, rn.F32)
    assert (p2.block_threads, p2.vecs_per_thread, p2.vec_bytes) == (256, 2, 16)


def test_huge_row_still_planned():
    # 8 MiB rows: the looped vector body, for decode and prefill row counts
    for rows in (4, 100000):
        rc, p = plan(rows, 1 << 22, rn.BF16)
        assert rc == rn.OK and p.vecs_per_thread == 0 and p.vec_bytes == 16, p.as_dict()
    # misaligned: the scalar body
    rc, p = plan(4, 1 << 22, rn.BF16, xoff=2)
    assert rc == rn.OK and p.variant == rn.VARIANT_GENERIC


def test_plan_struct_layout():
    assert ctypes.sizeof(rn.Plan) == 40


def test_per_kernel_parity_plans_are_valid():
    """The explicit plans the GPU per-kernel test launches all pass the
    library's own plan validation (checked here, host only)."""
    import sys
    sys.path.insert(0, os.path.dirname(__file__))
    import test_gpu_kernels as tk
    n = 0
    for k in rn.kernels():
        es = tk.ES[k["dtype"]]
        for hidden, pd in tk.plans_for(k, 37, SMS, OPTIN):
            rc = rn.rmsnorm_validate_plan_epilogue(rn.Plan(**pd), A, 3 * A, 5 * A, 37, hidden,
                                                   k["dtype"], k["epilogue"], SMS, OPTIN)
            assert rc == rn.OK, (k, hidden, pd, rc)
            n += 1
    assert n > 1000


def test_validation_rejects_bad_plans():
    rc, p = plan(64, 4096, rn.BF16, rn.VARIANT_CTA_PER_ROW)
    assert rc == rn.OK
    bad = rn.Plan(**p.as_dict())
    bad.block_threads = 33
    assert rn.rmsnorm_validate_plan(bad, A, 3 * A, 5 * A, 64, 4096, rn.BF16, SMS, OPTIN) != rn.OK
    bad = rn.Plan(**p.as_dict())
    bad.kernel_index = 10 ** 6
    assert rn.rmsnorm_validate_plan(bad, A, 3 * A, 5 * A, 64, 4096, rn.BF16, SMS, OPTIN) != rn.OK
    bad = rn.Plan(**p.as_dict())
    bad.block_threads = 32  # too few threads for the row
    assert rn.rmsnorm_validate_plan(bad, A, 3 * A, 5 * A, 64, 4096, rn.BF16, SMS, OPTIN) == \
        rn.ERR_VARIANT
    # a plan for another element type
    assert rn.rmsnorm_validate_plan(p, A, 3 * A, 5 * A, 64, 4096, rn.F16, SMS, OPTIN) != rn.OK
    rc, sp = plan(4096, 4096, rn.BF16, rn.VARIANT_STAGED)
    bad = rn.Plan(**sp.as_dict())
    bad.smem_bytes += 16
    assert rn.rmsnorm_validate_plan(bad, A, 3 * A, 5 * A, 4096, 4096, rn.BF16, SMS, OPTIN) != rn.OK
    bad = rn.Plan(**sp.as_dict())
    bad.stages += 1  # no longer a multiple of the consumer count
    assert rn.rmsnorm_validate_plan(bad, A, 3 * A, 5 * A, 4096, 4096, rn.BF16, SMS, OPTIN) != rn.OK


# ------------------------------------------------------------- QK norm validation (host only)

def qk(q, k, qw, kw, tokens, hq, hk, d, qs, ks, bias=0.0, eps=1e-6, dtype=rn.BF16):
    return rn._load().rmsnorm_qk_norm(q, k, qw, kw, tokens, hq, hk, d, qs, ks, bias, eps, dtype,
                                      None)


VALIDATED = (rn.ERR_CUDA, rn.ERR_NOT_INITIALIZED, rn.OK)  # got past argument checks


def test_qk_norm_argument_checks():
    Q, K, W = 1 << 40, 1 << 41, 1 << 42
    assert qk(Q, K, W, W, 4, 8, 2, 128, 0, 0) in VALIDATED
    assert qk(Q, K, W, W, 4, 8, 2, 128, 0, 0, dtype=9) == rn.ERR_UNSUPPORTED_DTYPE
    assert qk(Q, K, W, W, -1, 8, 2, 128, 0, 0) == rn.ERR_INVALID_ARG
    assert qk(Q, K, W, W, 4, 8, 2, 0, 0, 0) == rn.ERR_INVALID_ARG
    assert qk(Q, K, W, W, 4, 8, 2, 128, 8 * 128 - 1, 0) == rn.ERR_INVALID_ARG  # stride < heads
    assert qk(Q, K, W, W, 4, 8, 2, 128, 0, 0, eps=-1.0) == rn.ERR_INVALID_ARG
    assert qk(Q, K, W, W, 4, 8, 2, 128, 0, 0, bias=float("inf")) == rn.ERR_INVALID_ARG
    assert qk(0, K, W, W, 4, 8, 2, 128, 0, 0) == rn.ERR_INVALID_ARG
    assert qk(0, K, 0, W, 4, 0, 2, 128, 0, 0) in VALIDATED  # no q heads: q may be NULL


def test_qk_norm_fused_qkv_layout_accepted_overlaps_refused():
    B, W = 1 << 40, 1 << 42
    d, hq, hk, T = 128, 8, 2, 1000
    width = (hq + 2 * hk) * d
    es = 2
    # q at the token's start, k right after q, v after k: disjoint, accepted
    assert qk(B, B + hq * d * es, W, W, T, hq, hk, d, width, width) in VALIDATED
    # k starting inside the q heads: refused
    assert qk(B, B + (hq - 1) * d * es, W, W, T, hq, hk, d, width, width) == rn.ERR_ALIASING
    # k one token later but overlapping the next token's q heads: refused
    assert qk(B, B + width * es, W, W, T, hq, hk, d, width, width) == rn.ERR_ALIASING
    # a weight inside a q head: refused
    assert qk(B, B + hq * d * es, B + 5 * width * es + 64, W, T, hq, hk, d, width, width) == \
        rn.ERR_ALIASING
    # a weight in the v slot (not written): accepted
    assert qk(B, B + hq * d * es, B + (hq + hk) * d * es, W, T, hq, hk, d, width, width) in \
        VALIDATED


def test_qk_norm_overlap_rule_matches_brute_force():
    """The strided-overlap test inside rmsnorm_qk_norm against an explicit
    byte-set intersection on small random layouts (equal strides)."""
    import random
    rnd = random.Random(0)
    B, W = 1 << 40, 1 << 44
    for _ in range(400):
        d = rnd.choice([1, 2, 3, 8])
        hq, hk = rnd.randint(1, 3), rnd.randint(1, 3)
        T = rnd.randint(1, 5)
        stride = (hq + hk) * d + rnd.randint(0, 6)
        off = rnd.randint(-3 * stride, 3 * stride)
        qset = {t * stride + e for t in range(T) for e in range(hq * d)}
        kset = {off + t * stride + e for t in range(T) for e in range(hk * d)}
        collide = bool(qset & kset)
        rc = qk(B, B + 2 * off, W, W, T, hq, hk, d, stride, stride)
        assert (rc == rn.ERR_ALIASING) == collide, (d, hq, hk, T, stride, off, rc)


# ------------------------------------------------------------------ epilogues

def plan_epi(rows, hidden, dtype, epi, variant=rn.VARIANT_AUTO, x=None, w=None, y=None):
    return rn.rmsnorm_plan_epilogue_status(x or A, w or 3 * A, y or 5 * A, rows, hidden, dtype,
                                           epi, SMS, OPTIN, variant)


def test_epilogue_kernel_sets():
    ks = rn.kernels()
    for dt in (rn.F32, rn.BF16, rn.F16):
        plain = [k for k in ks if k["dtype"] == dt and k["epilogue"] == rn.EPI_PLAIN]
        bias = [k for k in ks if k["dtype"] == dt and k["epilogue"] == rn.EPI_BIAS]
        mx = [k for k in ks if k["dtype"] == dt and k["epilogue"] == rn.EPI_MXFP8]
        key = lambda k: (k["variant"], k["vec_bytes"], k["tpr"], k["nv"], k["block"],
                         k["min_blocks"], k["cache_policy"])
        # every register / looped / staged / generic body has a bias twin; the
        # cluster and grid ones have none
        assert {key(k) for k in bias} == {key(k) for k in plain
                                          if k["variant"] not in (rn.VARIANT_CLUSTER,
                                                                  rn.VARIANT_GRID)}
        # block-scaled outputs: the register and looped bodies except the 4-lane
        # group, the staged ring with register stores, and their own blocks of
        # a compile-time size with four 32-byte vectors per thread: one warp
        # (16 resident), 64, 96 and 128 threads (register-capped at 64)
        want = {key(k) for k in plain if (k["variant"] in (rn.VARIANT_WARP_PER_ROW,
                                                           rn.VARIANT_CTA_PER_ROW)
                                          and k["tpr"] != 4)
                or (k["variant"] == rn.VARIANT_STAGED and k["cache_policy"] != 3)}
        want |= {(rn.VARIANT_CTA_PER_ROW, 32, t, 4, t, 1024 // t, 1) for t in (64, 96, 128)}
        want.add((rn.VARIANT_CTA_PER_ROW, 32, 32, 4, 32, 16, 1))
        assert {key(k) for k in mx} == want
        for epi in (rn.EPI_MXFP4, rn.EPI_NVFP4):
            assert {key(k) for k in ks if k["dtype"] == dt and k["epilogue"] == epi} == want


@pytest.mark.parametrize("epi", [rn.EPI_BIAS, rn.EPI_MXFP8])
def test_epilogue_selector_matches_plain_bodies_outside_the_staged_range(epi):
    """The epilogues take the same body as the plain output wherever that is
    not the cluster split or the grid variant (block-scaled outputs: nor the
    1-32 KiB prefill rows, where they take their own shapes, nor the staged
    ring), and a kernel of their own epilogue."""
    ks = rn.kernels()
    for rows in (1, 8, 100, 152, 4096, 65536):
        for hidden in (128, 512, 1024, 2048, 4096, 8192, 16384, 20480, 36864, 65536, 131072):
            for dt in (rn.BF16, rn.F32):
                rc, p = plan_epi(rows, hidden, dt, epi)
                assert rc == rn.OK, (rows, hidden, dt, rc)
                assert ks[p.kernel_index]["epilogue"] == epi
                rc0, p0 = plan_epi(rows, hidden, dt, rn.EPI_PLAIN)
                nvec = hidden * (4 if dt == rn.F32 else 2) // 16
                if epi == rn.EPI_MXFP8 and rows > SMS and 64 < nvec <= 2048:
                    # block-scaled prefill rows of 1-32 KiB: their own shapes
                    # (a warp x two 32-byte vectors for 1-2 KiB rows on 4 blocks
                    # per SM, a one-warp block x four for 2-3 KiB rows, then
                    # 32-byte vectors, 2 or 4 per thread)
                    if nvec <= 128:
                        assert p.variant == rn.VARIANT_WARP_PER_ROW
                        assert (p.vec_bytes, p.vecs_per_thread) == (32, 2)
                        assert p.grid <= 4 * SMS
                    elif nvec <= 192:
                        k = ks[p.kernel_index]
                        assert (k["tpr"], k["nv"], p.vec_bytes, p.block_threads) == (32, 4, 32, 32)
                    else:
                        assert p.vec_bytes == 32 and p.vecs_per_thread in (2, 4)
                        if 256 < nvec <= 1024:
                            # the smallest compile-time block of 64 / 96 / 128
                            # threads x 4 vectors that holds the row
                            n32 = nvec // 2
                            tprc = 64 if n32 <= 256 else (96 if n32 <= 384 else 128)
                            k = ks[p.kernel_index]
                            assert (k["tpr"], k["nv"], k["min_blocks"]) == \
                                (tprc, 4, 1024 // tprc), (rows, hidden, dt, k)
                            assert p.block_threads == tprc
                        if 1536 < nvec <= 2048:
                            # 24-32 KiB rows, MXFP8: two vectors per thread on
                            # 2 blocks per SM
                            assert p.vecs_per_thread == 2 and p.grid <= 2 * SMS
                        if 1024 < nvec <= 1536:
                            # 16-24 KiB rows: the body capped at 96 registers,
                            # one block per row
                            k = ks[p.kernel_index]
                            assert (k["nv"], k["block"], k["min_blocks"]) == (4, 320, 2)
                            assert p.grid == rows
                    assert p.threads_per_row * p.vecs_per_thread * p.vec_bytes >= nvec * 16, \
                        (rows, hidden, dt, p.as_dict())
                    continue
                if epi == rn.EPI_MXFP8 and rows > SMS and nvec > 2048:
                    if nvec <= 2560:
                        # 32-40 KiB rows: the capped 32-byte four-vector body on
                        # 6 blocks per SM
                        k = ks[p.kernel_index]
                        assert (k["nv"], k["block"], k["min_blocks"]) == (4, 320, 2)
                        assert p.grid == min(rows, 6 * SMS)
                        continue
                    # longer rows: the looped body (not the ring, not the plain
                    # output's 32-byte blocks)
                    assert p.variant != rn.VARIANT_STAGED and p.vecs_per_thread == 0
                    continue
                row_bytes = nvec * 16
                if epi == rn.EPI_BIAS and rows > SMS and \
                        (16384 < row_bytes <= 24576 or 32768 < row_bytes <= 40960):
                    # the plain output's 32-byte four-vector blocks, in the
                    # build capped at 96 registers for the weight offset (two
                    # blocks of <= 320 threads per SM)
                    assert p0.vec_bytes == 32 and p0.vecs_per_thread == 4
                    assert (p.vec_bytes, p.vecs_per_thread, p.threads_per_row) == \
                        (32, 4, p0.threads_per_row)
                    k = ks[p.kernel_index]
                    assert (k["block"], k["min_blocks"]) == (320, 2)
                    continue
                if p0.variant not in (rn.VARIANT_CLUSTER, rn.VARIANT_GRID):
                    k, k0 = ks[p.kernel_index], ks[p0.kernel_index]
                    strip = lambda k: {a: b for a, b in k.items() if a not in ("index", "epilogue")}
                    assert strip(k) == strip(k0)
                    d, d0 = p.as_dict(), p0.as_dict()
                    d.pop("kernel_index"), d0.pop("kernel_index")
                    assert d == d0, (rows, hidden, dt)


def test_epilogue_argument_rules():
    # MXFP8 wants whole 32-element blocks and 16-byte vectors
    assert plan_epi(64, 4000, rn.BF16, rn.EPI_MXFP8)[0] == rn.OK      # 125 blocks
    assert plan_epi(64, 4008, rn.BF16, rn.EPI_MXFP8)[0] == rn.ERR_INVALID_ARG
    assert plan_epi(64, 4096, rn.BF16, rn.EPI_MXFP8, x=A + 2)[0] == rn.ERR_MISALIGNED
    assert plan_epi(64, 4096, rn.BF16, rn.EPI_MXFP8, y=A + 8)[0] == rn.ERR_MISALIGNED
    # the bias epilogue falls back to the scalar body like the plain one
    rc, p = plan_epi(64, 4097, rn.BF16, rn.EPI_BIAS)
    assert rc == rn.OK and p.variant == rn.VARIANT_GENERIC
    assert rn.kernels()[p.kernel_index]["epilogue"] == rn.EPI_BIAS
    # forced variants: the staged ring takes every output, the scalar body
    # no block-scaled one
    for epi in (rn.EPI_BIAS, rn.EPI_MXFP8, rn.EPI_NVFP4):
        rc, p = plan_epi(64, 4096, rn.BF16, epi, rn.VARIANT_STAGED)
        assert rc == rn.OK and rn.kernels()[p.kernel_index]["epilogue"] == epi
    assert plan_epi(64, 4096, rn.BF16, rn.EPI_MXFP8, rn.VARIANT_GENERIC)[0] == rn.ERR_VARIANT
    assert plan_epi(64, 4096, rn.BF16, 7)[0] == rn.ERR_INVALID_ARG
    # a plan naming another epilogue's kernel is refused
    rc, p = plan_epi(64, 4096, rn.BF16, rn.EPI_PLAIN)
    for epi in (rn.EPI_BIAS, rn.EPI_MXFP8):
        assert rn.rmsnorm_validate_plan_epilogue(p, A, 3 * A, 5 * A, 64, 4096, rn.BF16, epi,
                                                 SMS, OPTIN) == rn.ERR_INVALID_ARG


def test_epilogue_calls_validate_before_context():
    """Argument errors come before the context check (no GPU here)."""
    lib = rn._load()
    # hidden not a multiple of 32
    assert lib.rmsnorm_fwd_mxfp8(A, 3 * A, 5 * A, 7 * A, 4, 100, 0.0, 1e-6, rn.BF16,
                                 None) == rn.ERR_INVALID_ARG
    # non-finite bias
    assert lib.rmsnorm_fwd_bias(A, 3 * A, 5 * A, 4, 128, float("inf"), 1e-6, rn.BF16,
                                None) == rn.ERR_INVALID_ARG
    # scales overlapping the codes, codes overlapping x
    assert lib.rmsnorm_fwd_mxfp8(A, 3 * A, 5 * A, 5 * A + 64, 4, 128, 0.0, 1e-6, rn.BF16,
                                 None) == rn.ERR_ALIASING
    assert lib.rmsnorm_fwd_mxfp8(A, 3 * A, A + 256, 7 * A, 4, 128, 0.0, 1e-6, rn.BF16,
                                 None) == rn.ERR_ALIASING
    assert lib.rmsnorm_fwd_mxfp8(A, 3 * A, 5 * A, None, 4, 128, 0.0, 1e-6, rn.BF16,
                                 None) == rn.ERR_INVALID_ARG


# ------------------------------------------------------------------ cluster split

def test_cluster_plans():
    for rows, hidden, C in ((1, 65536, 8), (8, 16384, 4), (1, 4096, 2), (32, 32768, 8)):
        rc, p = plan(rows, hidden, rn.BF16, rn.VARIANT_CLUSTER)
        assert rc == rn.OK and p.variant == rn.VARIANT_CLUSTER and p.stages == C
        assert p.grid == rows * C and p.block_threads * p.vecs_per_thread * C * 16 >= hidden * 2
        assert rn.rmsnorm_validate_plan(p, A, 3 * A, 5 * A, rows, hidden, rn.BF16, SMS,
                                        OPTIN) == rn.OK
        bad = rn.Plan(**p.as_dict())
        bad.grid += 1                       # one cluster per row, exactly
        assert rn.rmsnorm_validate_plan(bad, A, 3 * A, 5 * A, rows, hidden, rn.BF16, SMS,
                                        OPTIN) == rn.ERR_VARIANT
        bad = rn.Plan(**p.as_dict())
        bad.stages = 3                      # cluster sizes 2, 4, 8
        assert rn.rmsnorm_validate_plan(bad, A, 3 * A, 5 * A, rows, hidden, rn.BF16, SMS,
                                        OPTIN) == rn.ERR_VARIANT
    # plain output only; vectors need alignment
    assert plan_epi(1, 65536, rn.BF16, rn.EPI_BIAS, rn.VARIANT_CLUSTER)[0] == rn.ERR_VARIANT
    assert plan(1, 65536, rn.BF16, rn.VARIANT_CLUSTER, xoff=2)[0] == rn.ERR_MISALIGNED
    # a stages value on a non-staged, non-cluster plan is refused
    rc, p = plan(64, 4096, rn.BF16, rn.VARIANT_CTA_PER_ROW)
    p.stages = 2
    assert rn.rmsnorm_validate_plan(p, A, 3 * A, 5 * A, 64, 4096, rn.BF16, SMS,
                                    OPTIN) == rn.ERR_INVALID_ARG


def test_cluster_split_chosen_for_long_decode_rows():
    ks = rn.kernels()
    for rows, hidden, C in ((1, 32768, 8), (1, 65536, 8), (8, 65536, 8), (19, 65536, 8),
                            (20, 65536, 4), (32, 32768, 4), (64, 32768, 2), (76, 32768, 2),
                            (1, 20480, 8), (8, 20480, 8), (32, 24576, 4)):
        rc, p = plan(rows, hidden, rn.BF16)
        assert rc == rn.OK and p.variant == rn.VARIANT_CLUSTER and p.stages == C, \
            (rows, hidden, p.as_dict())
        assert p.vec_bytes == 32 and p.block_threads <= 512
        assert ks[p.kernel_index]["variant"] == rn.VARIANT_CLUSTER
    # 64-256 KiB rows, up to 128 of them, more than one wave holds: clusters
    # over several waves (4 blocks below 128 KiB rows, 8 from there)
    for rows, hidden, C in ((77, 65536, 8), (48, 131072, 8), (80, 65536, 8), (96, 65536, 8),
                            (128, 65536, 8), (128, 131072, 8), (77, 40960, 4), (96, 40960, 4),
                            (128, 40960, 4), (128, 36864, 4)):
        rc, p = plan(rows, hidden, rn.BF16)
        assert rc == rn.OK and p.variant == rn.VARIANT_CLUSTER and p.stages == C, \
            (rows, hidden, p.as_dict())
        assert p.grid == rows * C > SMS and p.vecs_per_thread * p.vec_bytes >= 64
    # exactly 64 KiB rows: one wave of clusters while rows * 2 <= SMs; beyond
    # that the several-waves rule (rows above 64 KiB only) does not apply and
    # the block-per-row body keeps them
    for rows in (77, 96, 128):
        rc, p = plan(rows, 32768, rn.BF16)
        assert rc == rn.OK and p.variant == rn.VARIANT_PERSISTENT, (rows, p.as_dict())
    rc, p = plan(76, 32768, rn.BF16)
    assert rc == rn.OK and p.variant == rn.VARIANT_CLUSTER and p.stages == 2
    # 512 KiB rows: 16-byte vectors, four per thread, 1024 threads per block
    rc, p = plan(1, 131072, rn.F32)
    assert rc == rn.OK and p.variant == rn.VARIANT_CLUSTER and p.stages == 8
    assert p.vec_bytes == 16 and p.vecs_per_thread == 4 and p.block_threads == 1024
    # shorter rows, more rows than fit one block per SM, or an epilogue: no cluster
    for rows, hidden, epi in ((1, 16384, 0), (32, 16384, 0), (77, 32768, 0), (153, 65536, 0),
                              (9, 20480, 0), (32, 20480, 0), (48, 24576, 0), (129, 65536, 0),
                              (128, 32768, 0), (152, 131072, 0), (129, 40960, 0),
                              (1, 65536, rn.EPI_BIAS), (1, 65536, rn.EPI_MXFP8)):
        rc, p = plan_epi(rows, hidden, rn.BF16, epi)
        assert rc == rn.OK and p.variant != rn.VARIANT_CLUSTER, (rows, hidden, epi)



def test_fp4_argument_rules():
    assert plan_epi(64, 4096, rn.BF16, rn.EPI_MXFP4)[0] == rn.OK
    assert plan_epi(64, 4080, rn.BF16, rn.EPI_MXFP4)[0] == rn.ERR_INVALID_ARG
    assert plan_epi(64, 4080, rn.BF16, rn.EPI_NVFP4)[0] == rn.OK        # 255 blocks of 16
    assert plan_epi(64, 4088, rn.BF16, rn.EPI_NVFP4)[0] == rn.ERR_INVALID_ARG
    assert plan_epi(64, 4096, rn.BF16, rn.EPI_NVFP4, x=A + 2)[0] == rn.ERR_MISALIGNED
    assert plan_epi(64, 4096, rn.BF16, 5)[0] == rn.ERR_INVALID_ARG
    for epi in (rn.EPI_MXFP4, rn.EPI_NVFP4):   # the block-scaled shapes of MXFP8
        rc, p = plan_epi(16384, 4096, rn.BF16, epi)
        rc8, p8 = plan_epi(16384, 4096, rn.BF16, rn.EPI_MXFP8)
        d, d8 = p.as_dict(), p8.as_dict()
        d.pop("kernel_index"), d8.pop("kernel_index")
        assert rc == rn.OK and d == d8
    lib = rn._load()
    # codes are hidden / 2 bytes a row: scales right after the codes do not overlap
    assert lib.rmsnorm_fwd_mxfp4(A, 3 * A, 5 * A, 5 * A + 4 * 2048, 4, 4096, 0.0, 1e-6, rn.BF16,
                                 None) in (rn.ERR_NOT_INITIALIZED, rn.ERR_CUDA)  # past the checks
    assert lib.rmsnorm_fwd_mxfp4(A, 3 * A, 5 * A, 5 * A + 4 * 2048 - 1, 4, 4096, 0.0, 1e-6,
                                 rn.BF16, None) == rn.ERR_ALIASING
    assert lib.rmsnorm_fwd_nvfp4(A, 3 * A, 5 * A, 7 * A, 4, 4096, 0.0, 0.0, 1e-6, rn.BF16,
                                 None) == rn.ERR_INVALID_ARG



def test_grid_plans():
    # rows too long for a cluster: the grid variant, 2 blocks of 512 threads per SM
    for rows, hidden, dt in ((1, 1 << 20, rn.BF16), (8, 300000, rn.F32), (64, 262152, rn.BF16)):
        rc, p = plan(rows, hidden, dt)
        assert rc == rn.OK and p.variant == rn.VARIANT_GRID, (rows, hidden, p.as_dict())
        assert p.grid == (SMS if rows == 1 else 2 * SMS) and p.rows_per_block == rows
        assert p.block_threads == (256 if rows == 1 else 512)
        assert rn.rmsnorm_validate_plan(p, A, 3 * A, 5 * A, rows, hidden, dt, SMS,
                                        OPTIN) == rn.OK
        bad = rn.Plan(**p.as_dict())
        bad.grid = 2 * SMS + 1          # more blocks than the SMs hold at once
        assert rn.rmsnorm_validate_plan(bad, A, 3 * A, 5 * A, rows, hidden, dt, SMS,
                                        OPTIN) == rn.ERR_VARIANT
    # rows a cluster holds, more rows than 64, or an epilogue: not the grid variant
    assert plan(1, 1 << 18, rn.BF16)[1].variant == rn.VARIANT_CLUSTER
    assert plan(65, 1 << 20, rn.BF16, rn.VARIANT_GRID)[0] == rn.ERR_VARIANT
    assert plan_epi(1, 1 << 20, rn.BF16, rn.EPI_BIAS, rn.VARIANT_GRID)[0] == rn.ERR_VARIANT
    assert plan(1, 1 << 20, rn.BF16, rn.VARIANT_GRID, xoff=2)[0] == rn.ERR_MISALIGNED



def test_maximum_row_length_rule():
    assert plan(1, 1 << 26, rn.BF16)[0] == rn.OK
    assert plan(1, (1 << 26) + 8, rn.BF16)[0] == rn.ERR_INVALID_ARG
    assert plan(1, 1 << 26, rn.BF16)[1].variant == rn.VARIANT_GRID


@pytest.mark.parametrize("epi", ["plain", "bias", "mxfp8", "mxfp4", "nvfp4"])
def test_tuning_candidates_are_valid_plans(epi):
    """The plans the tuning sweep would time are well formed: the library's own
    plan check (host only) takes them, or refuses them only because the shape
    does not fit the body (the sweep skips those), for decode, mid, wide and
    very long rows."""
    from rmsnorm_fwd_gb300 import tune
    code = {"plain": 0, "bias": 1, "mxfp8": 2, "mxfp4": 3, "nvfp4": 4}[epi]
    n = 0
    for rows, hidden in ((1, 4096), (32, 65536), (8192, 1024), (16384, 4096), (4096, 24576),
                         (64, 262144), (1, 1 << 20)):
        for p in tune.candidates(rows, hidden, "bf16", SMS, OPTIN, code):
            rc = rn.rmsnorm_validate_plan_epilogue(rn.Plan(**p), A, 3 * A, 5 * A, rows, hidden,
                                                   rn.BF16, code, SMS, OPTIN)
            assert rc in (rn.OK, rn.ERR_VARIANT), (rows, hidden, p, rc)
            n += rc == rn.OK
    assert n > 50



def test_prefill_rows_of_16_to_24_and_32_to_40_kib_take_32_byte_blocks():
    for hidden in (10240, 12288, 18432, 20480):
        rc, p = plan(16384, hidden, rn.BF16)
        assert rc == rn.OK and p.variant == rn.VARIANT_CTA_PER_ROW and p.vec_bytes == 32
        assert p.vecs_per_thread == 4 and p.grid == 16384, (hidden, p.as_dict())
    assert plan(16384, 16384, rn.BF16)[1].variant == rn.VARIANT_PERSISTENT   # 32 KiB rows
    assert plan(16384, 24576, rn.BF16)[1].variant == rn.VARIANT_STAGED       # 48 KiB rows
    # the weight-offset output takes the same shape in its build capped at 96
    # registers (two blocks of <= 320 threads per SM)
    for hidden in (10240, 20480):
        rc, p = rn.rmsnorm_plan_epilogue_status(A, 3 * A, 5 * A, 16384, hidden, rn.BF16,
                                                rn.EPI_BIAS, SMS, OPTIN)
        assert rc == rn.OK and p.variant == rn.VARIANT_CTA_PER_ROW and p.vec_bytes == 32
        k = rn.kernels()[p.kernel_index]
        assert (k["nv"], k["block"], k["min_blocks"]) == (4, 320, 2)


def test_host_mapped_plan_caps_wide_row_grids_at_two_blocks_per_sm():
    """rmsnorm_fwd_host's page-locked path: block-per-row and wide persistent
    grids of the register bodies become two persistent blocks per SM; short
    batches, warp-per-row, staged and looped plans are rmsnorm_plan's."""
    def both(rows, hidden, dt=rn.BF16):
        rc, p = rn.rmsnorm_plan_host_mapped_status(A, 3 * A, 5 * A, rows, hidden, dt, SMS, OPTIN)
        rc0, p0 = plan(rows, hidden, dt)
        assert rc == rc0 == rn.OK
        return p, p0
    p, p0 = both(16384, 4096)
    assert p0.variant == rn.VARIANT_CTA_PER_ROW and p0.grid == 16384
    assert p.variant == rn.VARIANT_PERSISTENT and p.grid == 2 * SMS
    d, d0 = p.as_dict(), p0.as_dict()
    for k in ("variant", "grid"):
        d.pop(k), d0.pop(k)
    assert d == d0                                   # the same body and block
    assert rn.rmsnorm_validate_plan(p, A, 3 * A, 5 * A, 16384, 4096, rn.BF16, SMS, OPTIN) == rn.OK
    for rows, hidden in ((100, 4096), (2 * SMS, 4096), (16384, 512), (16384, 24576), (4, 131072)):
        p, p0 = both(rows, hidden)
        if p0.variant in (rn.VARIANT_CTA_PER_ROW, rn.VARIANT_PERSISTENT) and p0.grid > 2 * SMS:
            assert p.variant == rn.VARIANT_PERSISTENT and p.grid == 2 * SMS
        else:
            assert p.as_dict() == p0.as_dict(), (rows, hidden)
    assert rn.rmsnorm_plan_host_mapped_status(A, 3 * A, 5 * A, 8, 4096, 7, SMS, OPTIN)[0] == \
        rn.ERR_UNSUPPORTED_DTYPE
    # the same argument rules as rmsnorm_plan: zero rows plan nothing, a null
    # plan pointer or no SMs are refused
    assert rn.rmsnorm_plan_host_mapped_status(A, 3 * A, 5 * A, 0, 4096, rn.BF16, SMS,
                                              OPTIN)[0] == rn.OK
    assert rn._load().rmsnorm_plan_host_mapped(A, 3 * A, 5 * A, 8, 4096, rn.BF16, SMS, OPTIN,
                                               None) == rn.ERR_INVALID_ARG
    assert rn.rmsnorm_plan_host_mapped_status(A, 3 * A, 5 * A, 8, 4096, rn.BF16, 0,
                                              OPTIN)[0] == rn.ERR_INVALID_ARG


def test_looped_body_block_size_for_72_to_80_kib_rows():
    """Rows beyond the staged ring up to 80 KiB: 256-thread looped blocks in
    batches of more than two rows per SM, 512 threads below that."""
    for rows, threads in ((2 * SMS + 1, 256), (512, 256), (2 * SMS, 512), (256, 512),
                          (SMS + 1, 512)):
        rc, p = plan(rows, 40960, rn.BF16)
        assert rc == rn.OK and p.vecs_per_thread == 0 and p.block_threads == threads, \
            (rows, p.as_dict())
    rc, p = plan(256, 65536, rn.BF16)                # longer rows: 512 threads always
    assert rc == rn.OK and p.vecs_per_thread == 0 and p.block_threads == 512
    rc, p = plan_epi(256, 40960, rn.BF16, rn.EPI_MXFP8)   # block-scaled: unchanged
    assert rc == rn.OK and p.vecs_per_thread == 0 and p.block_threads == 256
