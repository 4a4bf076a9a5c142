"""Host-only properties of the selector on random shapes (no GPU): every plan
it returns -- automatic, forced, for any epilogue, and the host-buffer plan
-- passes the library's own plan validation and covers the row; refusals
are one of the documented statuses."""
import numpy as np
import pytest

import rmsnorm_fwd_gb300 as rn

SMS, OPTIN = 152, 232448
A = 1 << 30
ES = {rn.F32: 4, rn.BF16: 2, rn.F16: 2}
REFUSALS = {rn.ERR_VARIANT, rn.ERR_MISALIGNED, rn.ERR_INVALID_ARG}


def random_cases(n, seed):
    rng = np.random.default_rng(seed)
    for _ in range(n):
        dt = int(rng.choice([rn.F32, rn.BF16, rn.F16]))
        hidden = int(np.exp2(rng.uniform(0, 21)))
        if rng.random() < 0.5:
            hidden = max(16, hidden // 32 * 32)          # whole MX blocks half the time
        rows = int(np.exp2(rng.uniform(0, 17)))
        epi = int(rng.choice([rn.EPI_PLAIN, rn.EPI_BIAS, rn.EPI_MXFP8, rn.EPI_MXFP4,
                              rn.EPI_NVFP4]))
        xoff = int(rng.choice([0, 0, 0, 2, 16, 32]))
        yoff = int(rng.choice([0, 0, 0, 4, 16]))
        yield dt, rows, hidden, epi, xoff, yoff


def check_plan(p, dt, rows, hidden, epi, x, y):
    assert rn.rmsnorm_validate_plan_epilogue(p, x, 3 * A, y, rows, hidden, dt, epi, SMS,
                                             OPTIN) == rn.OK, p.as_dict()
    assert p.grid >= 1 and 32 <= p.block_threads <= 1024 and p.block_threads % 32 == 0
    if p.variant in (rn.VARIANT_CTA_PER_ROW, rn.VARIANT_PERSISTENT, rn.VARIANT_WARP_PER_ROW) \
            and p.vecs_per_thread > 0:
        # a register body holds the whole row
        assert p.threads_per_row * p.vecs_per_thread * p.vec_bytes >= hidden * ES[dt], \
            p.as_dict()
    if p.variant == rn.VARIANT_CLUSTER:
        assert p.grid == rows * p.stages and p.stages in (2, 4, 8)
        assert p.block_threads * p.vecs_per_thread * p.vec_bytes * p.stages >= hidden * ES[dt]


@pytest.mark.parametrize("seed", range(4))
def test_automatic_and_forced_plans_validate(seed):
    counts = {"auto": 0, "forced": 0, "refused": 0}
    for dt, rows, hidden, epi, xoff, yoff in random_cases(400, seed):
        x, y = A + xoff, 5 * A + yoff
        for v in range(0, 8):
            rc, p = rn.rmsnorm_plan_epilogue_status(x, 3 * A, y, rows, hidden, dt, epi, SMS,
                                                    OPTIN, v)
            if rc != rn.OK:
                assert rc in REFUSALS, (rc, dt, rows, hidden, epi, v)
                counts["refused"] += 1
                if v == rn.VARIANT_AUTO:
                    # the automatic choice refuses only what no body can do:
                    # block-scaled outputs of partial blocks or unaligned rows
                    assert epi in rn.QUANT_FORMATS, (rc, dt, rows, hidden, epi)
                continue
            check_plan(p, dt, rows, hidden, epi, x, y)
            counts["auto" if v == rn.VARIANT_AUTO else "forced"] += 1
    assert counts["auto"] > 180 and counts["forced"] > 450


@pytest.mark.parametrize("seed", range(2))
def test_host_mapped_plans_validate(seed):
    for dt, rows, hidden, _, xoff, yoff in random_cases(400, 100 + seed):
        x, y = A + xoff, 5 * A + yoff
        rc, p = rn.rmsnorm_plan_host_mapped_status(x, 3 * A, y, rows, hidden, dt, SMS, OPTIN)
        rc0, p0 = rn.rmsnorm_plan_status(x, 3 * A, y, rows, hidden, dt, SMS, OPTIN)
        assert rc == rc0
        if rc != rn.OK:
            continue
        check_plan(p, dt, rows, hidden, rn.EPI_PLAIN, x, y)
        assert p.grid <= max(p0.grid, 2 * SMS)


FIELDS = ("variant", "grid", "block_threads", "stages", "smem_bytes", "kernel_index",
          "threads_per_row", "rows_per_block")


@pytest.mark.parametrize("seed", range(3))
def test_validator_accepts_no_plan_that_breaks_its_body(seed):
    """Mutate one or two fields of the selector's plans at random: whatever
    rmsnorm_validate_plan_epilogue still accepts launches a body that covers
    the row with the block size its kernel allows (the checks a launch
    relies on to stay inside its buffers and its resources)."""
    rng = np.random.default_rng(1000 + seed)
    ks = rn.kernels()
    accepted = 0
    for dt, rows, hidden, epi, xoff, yoff in random_cases(300, 200 + seed):
        x, y = A + xoff, 5 * A + yoff
        rc, p0 = rn.rmsnorm_plan_epilogue_status(x, 3 * A, y, rows, hidden, dt, epi, SMS, OPTIN)
        if rc != rn.OK:
            continue
        for _ in range(12):
            d = p0.as_dict()
            for f in rng.choice(FIELDS, size=int(rng.integers(1, 3)), replace=False):
                if f == "kernel_index":
                    d[f] = int(rng.integers(-2, len(ks) + 2))
                elif f == "variant":
                    d[f] = int(rng.integers(-1, 9))
                elif f == "block_threads":
                    d[f] = int(rng.choice([0, 16, 32, 48, 64, 96, 128, 256, 288, 512, 640,
                                           1024, 1056, 2048]))
                elif f == "stages":
                    d[f] = int(rng.integers(-1, 10))
                else:
                    d[f] = int(rng.choice([-1, 0, 1, 2, 8, SMS, 2 * SMS, rows, rows * 4,
                                           rows + 1, 1 << 20]))
            p = rn.Plan(**d)
            if rn.rmsnorm_validate_plan_epilogue(p, x, 3 * A, y, rows, hidden, dt, epi, SMS,
                                                 OPTIN) != rn.OK:
                continue
            accepted += 1
            k = ks[p.kernel_index]
            assert k["dtype"] == dt and k["epilogue"] == epi
            assert p.grid >= 1 and 32 <= p.block_threads <= 1024 and p.block_threads % 32 == 0
            row_bytes = hidden * ES[dt]
            v = k["variant"]
            assert p.variant == v or (v == rn.VARIANT_CTA_PER_ROW and
                                      p.variant == rn.VARIANT_PERSISTENT)
            if v == rn.VARIANT_WARP_PER_ROW:
                assert p.block_threads == k["block"]
                assert k["tpr"] * k["nv"] * k["vec_bytes"] >= row_bytes
            elif v == rn.VARIANT_CTA_PER_ROW:
                assert p.block_threads <= k["block"]
                if k["nv"] > 0:
                    assert p.block_threads * k["nv"] * k["vec_bytes"] >= row_bytes
                if k["tpr"] > 0:
                    assert p.block_threads == k["tpr"]
            elif v == rn.VARIANT_CLUSTER:
                assert p.stages in (2, 4, 8) and p.grid == rows * p.stages
                assert p.block_threads <= k["block"]
                assert p.block_threads * k["nv"] * k["vec_bytes"] * p.stages >= row_bytes
            elif v == rn.VARIANT_GRID:
                assert rows <= 64 and p.grid <= 2 * SMS and p.rows_per_block == rows
            elif v == rn.VARIANT_STAGED:
                assert 1 <= p.grid <= rows and p.smem_bytes <= OPTIN and p.stages >= 1
            if v not in (rn.VARIANT_STAGED, rn.VARIANT_CLUSTER):
                assert p.stages == 0
            if v != rn.VARIANT_STAGED:
                assert p.smem_bytes == 0
    assert accepted > 100
