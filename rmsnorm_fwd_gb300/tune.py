"""Plan sweep for the RMSNorm kernels (the offline tuning behind the selector).

    python -m rmsnorm_fwd_gb300.tune --rows 16384 --hidden 4096 [--dtype bf16]
    python -m rmsnorm_fwd_gb300.tune --grid [--classes bulk,mid,decode]

For one shape, every feasible explicit plan (each compiled instantiation
with the block sizes, grid sizes and staged-ring shapes that make sense for
the row) is launched through rmsnorm_fwd_ex and timed with CUDA events over
back-to-back launches on rotating input/output sets larger than L2 (decode
shapes: replayed from a CUDA graph so host launch cost is excluded).  One
JSON line per plan, then the best plans.  --grid walks row sizes 128 B ..
64 KiB (bf16 hidden 64 .. 32768) for bulk (>= 256 MiB of input), mid (8192
rows) and decode (1, 8, 32, 128 rows) classes and prints, per point, the
best plans and the automatic plan's time.  Inputs are drawn on the device
(values do not affect timing).  Performance depends on row bytes, not on the
element type, so the grid runs bf16.
"""
from __future__ import annotations

import argparse
import json
import sys

L2 = 129 * 1024 * 1024
_AUTO_ONLY = False
GRID_HIDDEN = [64, 128, 256, 512, 768, 1024, 1536, 2048, 2560, 2880, 3072, 3584, 4096, 5120,
               6144, 7168, 8192, 10240, 12288, 16384, 24576, 32768]
ES = {"f32": 4, "bf16": 2, "f16": 2}


def staged_smem(row_bytes: int, stages: int) -> int:
    slot = (row_bytes + 127) // 128 * 128
    bar = ((2 * stages + 2) * 8 + 256 + 127) // 128 * 128
    return bar + slot * (stages + 1)


def candidates(rows: int, hidden: int, dtype: str, sms: int, optin: int,
               epi: int = 0) -> list[dict]:
    """Explicit plans worth timing for this shape and epilogue (the library
    validates each)."""
    import rmsnorm_fwd_gb300 as rn
    es = ES[dtype]
    dt = rn.DTYPE_CODES[dtype]
    out = []
    for k in rn.kernels():
        if k["dtype"] != dt or k["epilogue"] != epi:
            continue
        v = k["variant"]
        if v == rn.VARIANT_WARP_PER_ROW:
            vb = k["vec_bytes"]
            nvec = hidden * es // vb
            if hidden * es % vb or k["tpr"] * k["nv"] < nvec or k["tpr"] * k["nv"] >= 2 * nvec + 32:
                continue
            gpb = k["block"] // k["tpr"]
            full = -(-rows // gpb)
            for g in sorted({full, min(full, sms * 4), min(full, sms * 8), min(full, sms * 16)}):
                out.append(dict(variant=v, vec_bytes=vb, threads_per_row=k["tpr"],
                                vecs_per_thread=k["nv"], block_threads=k["block"],
                                rows_per_block=gpb, stages=0, grid=g, smem_bytes=0,
                                kernel_index=k["index"]))
        elif v == rn.VARIANT_CTA_PER_ROW:
            vb = k["vec_bytes"]
            if hidden * es % vb:
                continue
            nvec = hidden * es // vb
            if k["nv"] == 0:  # looped body: any row length
                for tpr in (256, 512):
                    for g in sorted({rows, min(rows, sms), min(rows, 2 * sms)}):
                        out.append(dict(variant=v if g == rows else rn.VARIANT_PERSISTENT,
                                        vec_bytes=vb, threads_per_row=tpr, vecs_per_thread=0,
                                        block_threads=tpr, rows_per_block=1, stages=0, grid=g,
                                        smem_bytes=0, kernel_index=k["index"]))
                continue
            tpr = max(32, -(-(-(-nvec // k["nv"])) // 32) * 32)
            if k["tpr"]:
                if k["tpr"] * k["nv"] < nvec or k["tpr"] * k["nv"] >= 2 * nvec + 32:
                    continue
                tpr = k["tpr"]
            if tpr > k["block"]:
                continue
            grids = {rows}
            for m in (1, 2, 3, 4, 6, 8, 16):
                if tpr * m <= 2048:
                    grids.add(min(rows, sms * m))
            for g in sorted(grids):
                out.append(dict(variant=v if g == rows else rn.VARIANT_PERSISTENT, vec_bytes=vb,
                                threads_per_row=tpr, vecs_per_thread=k["nv"], block_threads=tpr,
                                rows_per_block=1, stages=0, grid=g, smem_bytes=0,
                                kernel_index=k["index"]))
        elif v == rn.VARIANT_STAGED:
            rb = hidden * es
            if rb % 16:
                continue
            for bps in (1, 2):
                budget = min(optin, 233472 // bps - 1024)
                smax = 0
                for st in range(32, 0, -1):
                    if staged_smem(rb, st) <= budget:
                        smax = st
                        break
                for wpr, c in ((1, 2), (1, 4), (1, 6), (1, 8), (1, 12), (2, 2), (2, 4), (2, 6),
                               (4, 1), (4, 2), (4, 3), (8, 1), (8, 2), (16, 1)):
                    if c > smax:
                        continue
                    for st in sorted({smax // c * c, min(smax // c * c, 2 * c), c}):
                        if st < 2 or st % c:
                            continue
                        out.append(dict(variant=v, vec_bytes=16, threads_per_row=32 * wpr,
                                        vecs_per_thread=0, block_threads=32 * (c * wpr + 1),
                                        rows_per_block=c, stages=st, grid=min(rows, sms * bps),
                                        smem_bytes=staged_smem(rb, st), kernel_index=k["index"]))
        elif v == rn.VARIANT_CLUSTER:
            vb = k["vec_bytes"]
            if hidden * es % vb or (rows > 4 * sms and hidden * es < 16384):
                continue
            nvec = hidden * es // vb
            for C in (2, 4, 8):
                S = -(-nvec // C)
                tpr = max(32, -(-(-(-S // k["nv"])) // 32) * 32)
                if tpr > 1024 or (k["nv"] > 1 and tpr < 64):
                    continue
                out.append(dict(variant=v, vec_bytes=vb, threads_per_row=tpr * C,
                                vecs_per_thread=k["nv"], block_threads=tpr, rows_per_block=1,
                                stages=C, grid=rows * C, smem_bytes=0, kernel_index=k["index"]))
        elif v == rn.VARIANT_GRID:
            if hidden * es % 16 or rows > 64:
                continue
            for g in (sms, 2 * sms):
                for b in (256, 512):
                    out.append(dict(variant=v, vec_bytes=16, threads_per_row=b * g,
                                    vecs_per_thread=0, block_threads=b, rows_per_block=rows,
                                    stages=0, grid=g, smem_bytes=0, kernel_index=k["index"]))
        elif v == rn.VARIANT_GENERIC:
            for b in (256, 512, 1024):
                out.append(dict(variant=v, vec_bytes=0, threads_per_row=b, vecs_per_thread=0,
                                block_threads=b, rows_per_block=1, stages=0,
                                grid=min(rows, sms * (2048 // b)), smem_bytes=0,
                                kernel_index=k["index"]))
    return out


def time_plans(rows: int, hidden: int, dtype: str, iters: int, graph: bool,
               epi: int = 0, bias: float | None = None, host: bool = False) -> list[dict]:
    """Time the automatic plan and every candidate; sorted fastest first.
    epi: the epilogue (0 plain, 1 weight bias, 2-4 MXFP8 / MXFP4 / NVFP4
    output); bias: its weight offset (default 1.0 for the weight-bias output,
    -0.0 -- no offset, the exact-product form of 16-bit inputs -- for the
    block-scaled ones).  host: x and y in page-locked host memory (the
    kernel reads and writes it over the CPU-GPU link; plain output), the
    automatic plan being rmsnorm_fwd_host's (rmsnorm_plan_host_mapped)."""
    if bias is None:
        bias = 1.0 if epi == 1 else -0.0
    if host and epi != 0:
        raise ValueError("host buffers: the plain output only")
    import torch

    import rmsnorm_fwd_gb300 as rn
    dev = torch.device("cuda", 0)
    rn.ensure_context(0)
    sms, optin = rn.rmsnorm_device_limits()
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[dtype]
    es = ES[dtype]
    set_bytes = 2 * rows * hidden * es
    nsets = 2 if host else min(64, max(2, -(-3 * L2 // set_bytes)))
    if host:
        base = [torch.randn(rows, hidden).to(tdt).pin_memory() for _ in range(nsets)]
        xs = base
    else:
        base = [torch.randn(rows, hidden, device=dev).to(tdt) for _ in range(min(nsets, 4))]
        xs = [base[i % len(base)] if i < len(base) else base[i % len(base)].clone()
              for i in range(nsets)]
    mx = epi in rn.QUANT_FORMATS
    block, bits = rn.QUANT_FORMATS.get(epi, (1, 8 * es))
    if mx:
        ys = [torch.empty(rows * hidden * bits // 8, dtype=torch.uint8, device=dev)
              for _ in range(nsets)]
        ss = [torch.empty(rows * hidden // block, dtype=torch.uint8, device=dev)
              for _ in range(nsets)]
        sp = [t.data_ptr() for t in ss]
    else:
        ys = [torch.empty_like(xs[0]).pin_memory() if host else torch.empty_like(xs[0])
              for _ in range(nsets)]
        sp = [None] * nsets
    w = (1 + 0.1 * torch.randn(hidden, device=dev)).to(tdt)
    lib = rn._load()
    s = torch.cuda.current_stream().cuda_stream
    dt = rn.DTYPE_CODES[dtype]
    xp = [t.data_ptr() for t in xs]
    yp = [t.data_ptr() for t in ys]

    def fwd(x, wp, y, rows_, hidden_, eps, dt_, stream, variant, ref, j=0):
        if epi == 0:
            return lib.rmsnorm_fwd_ex(x, wp, y, rows_, hidden_, eps, dt_, stream, variant, ref)
        return lib.rmsnorm_fwd_epilogue_ex(x, wp, y, sp[j], rows_, hidden_, epi, bias, 0.01, eps,
                                           dt_, stream, variant, ref)

    auto = rn.Plan()
    if host:
        rc, auto = rn.rmsnorm_plan_host_mapped_status(xp[0], w.data_ptr(), yp[0], rows, hidden,
                                                      dt, sms, optin)
        if rc != rn.OK:
            raise rn.RmsnormError(rc, "rmsnorm_plan_host_mapped")
    else:
        fwd(xp[0], w.data_ptr(), yp[0], rows, hidden, 1e-6, dt, s, 0, rn.ctypes.byref(auto))
    cands = [auto.as_dict()] + ([] if _AUTO_ONLY else candidates(rows, hidden, dtype, sms, optin,
                                                                  epi))
    out_bytes = rows * hidden * bits // 8 + rows * hidden // block if mx else rows * hidden * es
    out = []
    for ci, c in enumerate(cands):
        p = rn.Plan(**c)
        ref = rn.ctypes.byref(p)
        if fwd(xp[0], w.data_ptr(), yp[0], rows, hidden, 1e-6, dt, s, 0, ref) != 0:
            continue
        for i in range(5):
            fwd(xp[i % nsets], w.data_ptr(), yp[i % nsets], rows, hidden, 1e-6, dt, s, 0, ref,
                i % nsets)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        if graph:
            g_ = torch.cuda.CUDAGraph()
            cs = torch.cuda.Stream()
            with torch.cuda.graph(g_, stream=cs):
                for i in range(iters):
                    fwd(xp[i % nsets], w.data_ptr(), yp[i % nsets], rows, hidden, 1e-6, dt,
                        cs.cuda_stream, 0, ref, i % nsets)
            g_.replay()
            torch.cuda.synchronize()
            e0.record()
            g_.replay()
            e1.record()
        else:
            e0.record()
            for i in range(iters):
                fwd(xp[i % nsets], w.data_ptr(), yp[i % nsets], rows, hidden, 1e-6, dt, s, 0, ref,
                    i % nsets)
            e1.record()
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) / iters * 1e3
        gbs = (rows * hidden * es + hidden * es + out_bytes) / (us * 1e-6) / 1e9
        out.append({"us": round(us, 3), "GBps": round(gbs, 1), "auto": ci == 0, "plan": c})
    del xs, ys, base
    torch.cuda.empty_cache()
    if rn.rmsnorm_get_device_status() != rn.OK:
        raise RuntimeError("a timed plan recorded a device-side error")
    out.sort(key=lambda r: r["us"])
    return out


def time_qk_plans(name: str, iters: int, graph: bool) -> list[dict]:
    """Every compiled QK-norm launch shape (lanes per head, vectors per lane,
    heads per group) x grid sizes on a QK workload (fused layout, rotating
    buffers larger than L2); sorted fastest first, the automatic plan marked."""
    import torch

    import rmsnorm_fwd_gb300 as rn
    from rmsnorm_fwd_gb300 import inputs
    wl = inputs.QK_WORKLOADS[name]
    rn.ensure_context(0)
    sms, _ = rn.rmsnorm_device_limits()
    dev = torch.device("cuda", 0)
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[wl.dtype]
    es = ES[wl.dtype]
    nbytes = wl.tokens * wl.width * es
    nsets = min(64, max(2, -(-3 * L2 // nbytes)))
    bufs = [torch.randn(wl.tokens * wl.width, device=dev).to(tdt) for _ in range(nsets)]
    qw = torch.ones(wl.head_dim, device=dev, dtype=tdt)
    d, hq, hk, T = wl.head_dim, wl.q_heads, wl.k_heads, wl.tokens
    fn = rn._load().rmsnorm_qk_norm_ex
    s = torch.cuda.current_stream().cuda_stream
    dt = rn.DTYPE_CODES[wl.dtype]
    ptr = [b.data_ptr() for b in bufs]
    auto = rn.QkPlan()
    rn.rmsnorm_qk_norm_ex(ptr[0], ptr[0] + hq * d * es, qw.data_ptr(), qw.data_ptr(), T, hq, hk,
                          d, wl.width, wl.width, 0.0, wl.eps, dt, s, auto)
    total = T * (hq + hk)
    cands = [auto.as_dict()]
    for lanes in (4, 8, 16, 32):
        for nv in (1, 2, 4):
            for rpg in (1, 2, 4):
                per = (256 // lanes) * rpg
                full = -(-total // per)
                for g in sorted({full, min(full, sms * 16), min(full, sms * 8), min(full, sms * 4)}):
                    cands.append(dict(lanes_per_head=lanes, vecs_per_lane=nv, heads_per_group=rpg,
                                      grid=g))
    out = []
    for ci, c in enumerate(cands):
        p = rn.QkPlan(**c)
        ref = rn.ctypes.byref(p)

        def call(i):
            return fn(ptr[i % nsets], ptr[i % nsets] + hq * d * es, qw.data_ptr(), qw.data_ptr(),
                      T, hq, hk, d, wl.width, wl.width, 0.0, wl.eps, dt, s, ref)
        if call(0) != 0:
            continue
        for i in range(5):
            call(i)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        if graph:
            g_ = torch.cuda.CUDAGraph()
            cs = torch.cuda.Stream()
            with torch.cuda.graph(g_, stream=cs):
                for i in range(iters):
                    fn(ptr[i % nsets], ptr[i % nsets] + hq * d * es, qw.data_ptr(), qw.data_ptr(),
                       T, hq, hk, d, wl.width, wl.width, 0.0, wl.eps, dt, cs.cuda_stream, ref)
            g_.replay()
            torch.cuda.synchronize()
            e0.record()
            g_.replay()
            e1.record()
        else:
            e0.record()
            for i in range(iters):
                call(i)
            e1.record()
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) / iters * 1e3
        out.append({"us": round(us, 3), "GBps": round(wl.bytes_per_call / (us * 1e-6) / 1e9, 1),
                    "auto": ci == 0, "plan": c})
    if rn.rmsnorm_get_device_status() != rn.OK:
        raise RuntimeError("a timed plan recorded a device-side error")
    out.sort(key=lambda r: r["us"])
    return out


def plan_label(p: dict, kinfo: dict) -> str:
    """Short text for a plan: variant, vector bytes, threads/row, vectors/thread,
    block, grid, stages, register floor, cache policy."""
    v = {1: "warp", 2: "block", 3: "staged", 4: "persistent", 5: "generic",
         6: "cluster", 7: "grid"}[p["variant"]]
    k = kinfo[p["kernel_index"]]
    nv = p["vecs_per_thread"] if p["variant"] != 3 else 0
    extra = f" W{p['threads_per_row'] // 32}" if p["variant"] == 3 else f" {nv}v"
    return (f"{v} {p['vec_bytes']}B{extra} t{p['threads_per_row']} b{p['block_threads']} "
            f"g{p['grid']}" + (f" st{p['stages']}" if p["stages"] else "")
            + (f" mb{k['min_blocks']}" if k["min_blocks"] else "")
            + (f" cp{k['cache_policy']}" if k["cache_policy"] else ""))


def summarize(path: str) -> str:
    """Markdown table of a --grid run: per point the best plan and the
    automatic plan."""
    import rmsnorm_fwd_gb300 as rn
    kinfo = {k["index"]: k for k in rn.kernels()}
    lines = ["| bf16 hidden (row bytes) | class | rows | best us | best GB/s | best plan | "
             "auto us | auto GB/s | auto / best |", "|" + "---|" * 9]
    for line in open(path):
        r = json.loads(line)
        b, a = r["top"][0], r["auto"]
        lines.append(f"| {r['hidden_bf16']} ({r['row_bytes']}) | {r['class']} | {r['rows']} | "
                     f"{b['us']:.2f} | {b['GBps']:.0f} | {plan_label(b['plan'], kinfo)} | "
                     f"{a['us']:.2f} | {a['GBps']:.0f} | {a['us'] / b['us']:.3f} |")
    return "\n".join(lines)


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--rows", type=int, default=16384)
    ap.add_argument("--hidden", type=int, default=4096)
    ap.add_argument("--dtype", default="bf16", choices=sorted(ES))
    ap.add_argument("--iters", type=int, default=100)
    ap.add_argument("--graph", action="store_true", help="replay launches from a CUDA graph")
    ap.add_argument("--grid", action="store_true", help="walk the row-size grid")
    ap.add_argument("--classes", default="bulk,mid,decode")
    ap.add_argument("--grid-hidden", default="", help="comma-separated bf16 hidden sizes")
    ap.add_argument("--keep", type=int, default=5)
    ap.add_argument("--pdl", type=int, choices=[0, 1], default=None,
                    help="programmatic dependent launch off/on (default: library setting)")
    ap.add_argument("--auto-only", action="store_true", help="time only the automatic plan")
    ap.add_argument("--summarize", default="", help="print a markdown table of a --grid output")
    ap.add_argument("--qk-workload", default="", help="sweep the QK-norm launch shapes instead")
    ap.add_argument("--epilogue", default="plain",
                    choices=["plain", "bias", "mxfp8", "mxfp4", "nvfp4"])
    ap.add_argument("--host-buffers", action="store_true",
                    help="x and y in page-locked host memory (plain output)")
    ap.add_argument("--weight-bias", type=float, default=None,
                    help="weight offset of the epilogue (default 1.0 for bias, -0.0 = none for "
                         "the block-scaled outputs)")
    args = ap.parse_args(argv)
    if args.qk_workload:
        if args.pdl is not None:
            import rmsnorm_fwd_gb300 as rn
            rn.rmsnorm_set_pdl(bool(args.pdl))
        for r in time_qk_plans(args.qk_workload, args.iters, args.graph)[:args.keep]:
            print(json.dumps(r), flush=True)
        return 0
    if args.summarize:
        print(summarize(args.summarize))
        return 0
    if args.pdl is not None:
        import rmsnorm_fwd_gb300 as rn
        rn.rmsnorm_set_pdl(bool(args.pdl))
    global _AUTO_ONLY
    _AUTO_ONLY = args.auto_only
    epi = {"plain": 0, "bias": 1, "mxfp8": 2, "mxfp4": 3, "nvfp4": 4}[args.epilogue]
    if not args.grid:
        res = time_plans(args.rows, args.hidden, args.dtype, args.iters, args.graph, epi,
                         args.weight_bias, args.host_buffers)
        for r in res:
            print(json.dumps(r), flush=True)
        return 0
    hidden = [int(h) for h in args.grid_hidden.split(",")] if args.grid_hidden else GRID_HIDDEN
    classes = args.classes.split(",")
    for h in hidden:
        points = []
        if "bulk" in classes:
            points.append(("bulk", max(4096, (256 << 20) // (2 * h)), 30, False))
        if "mid" in classes:
            points.append(("mid", 8192, 100, False))
        if "decode" in classes:
            points += [(f"decode{r}", r, 200, True) for r in (1, 8, 32, 128)]
        for cls, rows, iters, graph in points:
            res = time_plans(rows, h, "bf16", iters, graph, epi, args.weight_bias)
            auto = next((r for r in res if r["auto"]), None)
            print(json.dumps({"hidden_bf16": h, "row_bytes": 2 * h, "rows": rows, "class": cls,
                              "top": res[:args.keep], "auto": auto}), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
