"""Every compiled kernel instantiation, launched with explicit plans through
rmsnorm_fwd_ex (plain) or rmsnorm_fwd_epilogue_ex (weight bias, MXFP8, MXFP4, NVFP4),
against the fp64 oracle: full and partly filled rows, one row per block and
grid-stride (fewer blocks than rows), odd row counts."""
import pytest

import rmsnorm_fwd_gb300 as rn
from rmsnorm_fwd_gb300 import inputs

from _parity import compare, compare_quant, from_device, to_device

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

DT_NAME = {rn.F32: "f32", rn.BF16: "bf16", rn.F16: "f16"}
ES = {rn.F32: 4, rn.BF16: 2, rn.F16: 2}


@pytest.fixture(scope="module", autouse=True)
def ctx():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    rn.ensure_context(0)
    yield
    torch.cuda.synchronize()
    assert rn.rmsnorm_get_device_status() == rn.OK


def layout_bytes(row_bytes, stages):
    slot = (row_bytes + 127) // 128 * 128
    bar = ((2 * stages + 2) * 8 + 256 + 127) // 128 * 128
    return bar + slot * (stages + 1)


def plans_for(k, rows, sms, optin):
    """(hidden, plan dict) cases exercising kernel k.  MXFP8 kernels get
    row lengths of whole 32-element blocks."""
    cases = _plans_for(k, rows, sms, optin)
    if k["epilogue"] not in rn.QUANT_FORMATS:
        return cases
    block = rn.QUANT_FORMATS[k["epilogue"]][0]
    out = []
    for hidden, pd in cases:
        h = hidden // block * block
        if h == 0:
            h = block
        if pd["variant"] == rn.VARIANT_STAGED:   # the ring's layout follows the row length
            pd = dict(pd, smem_bytes=layout_bytes(h * ES[k["dtype"]], pd["stages"]))
            if pd["smem_bytes"] > optin:
                continue
        if pd["vecs_per_thread"] and h // (k["vec_bytes"] // ES[k["dtype"]]) > \
                pd["threads_per_row"] * pd["vecs_per_thread"]:
            continue
        out.append((h, pd))
    return list({(h, tuple(sorted(pd.items()))): (h, pd) for h, pd in out}.values())


def _plans_for(k, rows, sms, optin):
    es = ES[k["dtype"]]
    v = k["variant"]
    out = []
    if v == rn.VARIANT_WARP_PER_ROW:
        vpe = k["vec_bytes"] // es
        cap = k["tpr"] * k["nv"]
        for nvec in sorted({cap, max(1, cap - k["tpr"] + 1), max(1, cap // 2 + 1)}):
            gpb = k["block"] // k["tpr"]
            full = -(-rows // gpb)
            for grid in sorted({full, max(1, full // 3)}):
                out.append((nvec * vpe, dict(variant=v, vec_bytes=k["vec_bytes"],
                                             threads_per_row=k["tpr"], vecs_per_thread=k["nv"],
                                             block_threads=k["block"], rows_per_block=gpb,
                                             stages=0, grid=grid, smem_bytes=0,
                                             kernel_index=k["index"])))
    elif v == rn.VARIANT_CTA_PER_ROW and k["nv"] == 0:  # looped: any row length
        vpe = k["vec_bytes"] // es
        for tpr in (32, 96, k["block"]):
            for nvec in (1, tpr - 1, 4 * tpr + 3, 9 * tpr + 5):
                for grid in sorted({rows, max(1, rows // 4)}):
                    out.append((nvec * vpe, dict(variant=v if grid == rows else
                                                 rn.VARIANT_PERSISTENT,
                                                 vec_bytes=k["vec_bytes"], threads_per_row=tpr,
                                                 vecs_per_thread=0, block_threads=tpr,
                                                 rows_per_block=1, stages=0, grid=grid,
                                                 smem_bytes=0, kernel_index=k["index"])))
    elif v == rn.VARIANT_CTA_PER_ROW:
        vpe = k["vec_bytes"] // es
        tprs = [k["tpr"]] if k["tpr"] else sorted({32, 96, min(k["block"], 256), k["block"]})
        for tpr in tprs:
            for nvec in sorted({tpr * k["nv"], max(1, tpr * (k["nv"] - 1) + 1)}):
                for grid in sorted({rows, max(1, rows // 4)}):
                    out.append((nvec * vpe, dict(variant=v if grid == rows else
                                                 rn.VARIANT_PERSISTENT,
                                                 vec_bytes=k["vec_bytes"], threads_per_row=tpr,
                                                 vecs_per_thread=k["nv"], block_threads=tpr,
                                                 rows_per_block=1, stages=0, grid=grid,
                                                 smem_bytes=0, kernel_index=k["index"])))
    elif v == rn.VARIANT_STAGED:
        for hidden in (8 * 16 // es * 3, 4096 if es == 2 else 2048, 7168 if es == 2 else 3584,
                       20000 if es == 2 else 10000):
            rb = hidden * es
            for wpr, groups in ((1, 1), (1, 2), (1, 4), (2, 2), (4, 1), (4, 3), (8, 2)):
                stages = 2 * groups if k["cache_policy"] == 3 else groups
                for st in (stages, 2 * stages):
                    smem = layout_bytes(rb, st)
                    if smem > optin:
                        continue
                    for grid in sorted({min(rows, sms), max(1, rows // 5)}):
                        out.append((hidden, dict(variant=v, vec_bytes=16,
                                                 threads_per_row=32 * wpr, vecs_per_thread=0,
                                                 block_threads=32 * (groups * wpr + 1),
                                                 rows_per_block=groups, stages=st, grid=grid,
                                                 smem_bytes=smem, kernel_index=k["index"])))
    elif v == rn.VARIANT_CLUSTER:
        vpe = k["vec_bytes"] // es
        for C in (2, 4, 8):
            for tpr in (32, 160, 512):
                S = tpr * k["nv"]                       # a full slice per block
                for nvec in sorted({S * C, S * (C - 1) + 1, max(1, S * C - tpr + 3), 3}):
                    out.append((nvec * vpe, dict(variant=v, vec_bytes=k["vec_bytes"],
                                                 threads_per_row=tpr * C,
                                                 vecs_per_thread=k["nv"], block_threads=tpr,
                                                 rows_per_block=1, stages=C, grid=rows * C,
                                                 smem_bytes=0, kernel_index=k["index"])))
    elif v == rn.VARIANT_GRID:
        vpe = 16 // es
        for grid in (sms, 2 * sms, 7):
            for block in (64, 512):
                for nvec in (1, grid - 1, grid * 4 + 3, 40000):
                    out.append((nvec * vpe, dict(variant=v, vec_bytes=16,
                                                 threads_per_row=block * grid,
                                                 vecs_per_thread=0, block_threads=block,
                                                 rows_per_block=rows, stages=0, grid=grid,
                                                 smem_bytes=0, kernel_index=k["index"])))
    elif v == rn.VARIANT_GENERIC:
        for hidden in (1, 33, 1000, 4097):
            for block in (32, 256):
                out.append((hidden, dict(variant=v, vec_bytes=0, threads_per_row=block,
                                         vecs_per_thread=0, block_threads=block,
                                         rows_per_block=1, stages=0, grid=max(1, rows // 3),
                                         smem_bytes=0, kernel_index=k["index"])))
    return out


KERNELS = None


def kernel_ids():
    global KERNELS
    if KERNELS is None:
        KERNELS = rn.kernels()
    return [k["index"] for k in KERNELS]


@pytest.mark.parametrize("index", list(range(rn.rmsnorm_kernel_count())))
def test_kernel_instantiation(index):
    k = rn.kernels()[index]
    sms, optin = rn.rmsnorm_device_limits()
    rows = 37
    dt = DT_NAME[k["dtype"]]
    cases = plans_for(k, rows, sms, optin)
    assert cases, k
    epi = k["epilogue"]
    for hidden, pd in cases:
        x_np, w_np = inputs.random_case(rows, hidden, dt, seed=index)
        x = to_device(x_np, dt)
        w = to_device(w_np, dt)
        if epi in rn.QUANT_FORMATS:
            block, bits = rn.QUANT_FORMATS[epi]
            fmt = rn.EPI_NAMES[epi]
            # both instantiations of a 16-bit body: weight offset 0.625, and
            # -0 (no offset: the exact-product form)
            for bias in (0.625, -0.0):
                q = torch.full((rows, hidden * bits // 8), 0xAA, dtype=torch.uint8,
                               device="cuda")
                sc = torch.full((rows, hidden // block), 0xAA, dtype=torch.uint8, device="cuda")
                rn.rms_norm_quant(x, w, 1e-6, fmt, weight_bias=bias, global_scale=0.01, out=q,
                                  scales=sc, plan=rn.Plan(**pd))
                torch.cuda.synchronize()
                compare_quant(q.cpu().numpy(), sc.cpu().numpy(), x_np, w_np, bias, 1e-6, dt, fmt,
                              0.01)
            continue
        y = torch.full_like(x, 3.0)
        if epi == rn.EPI_BIAS:
            rn.rms_norm_bias(x, w, 0.625, 1e-6, out=y, plan=rn.Plan(**pd))
        else:
            rn.rms_norm(x, w, 1e-6, out=y, plan=rn.Plan(**pd))
        torch.cuda.synchronize()
        compare(from_device(y, dt), x_np, w_np, 1e-6, dt,
                bias=0.625 if epi == rn.EPI_BIAS else None)
