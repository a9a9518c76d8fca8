"""Small, self-contained launch sequence of one kernel for ncu captures.

    python -m mxfp8_block_scaled_moe_gb300.profile_case --kernel gemm1 --iters 3
    python -m mxfp8_block_scaled_moe_gb300.profile_case --kernel linear \
        --config qwen3_8b_down_prefill --iters 3

Builds one layer's inputs (default: the 16K-token Qwen3-30B-A3B-shaped
prefill), runs the routing step once, then launches the chosen kernel
``--iters`` times.  ``--kernel linear`` takes a dense-linear shape instead and
runs the whole linear call (activation quant + GEMM) ``--iters`` times;
``--kernel layer --fmt w4a8|w4a4`` runs the MXFP4-weight layers.  It holds about 1-2 GB on the device, more than the L2, so
DRAM counters are meaningful, and it launches only a few kernels before the
captured ones.
"""

from __future__ import annotations

import argparse

import torch

from . import api as mm
from . import workloads


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--config", default="qwen3_30b_prefill")
    ap.add_argument("--kernel", default="gemm1",
                    choices=["gemm1", "gemm2", "route", "finalize", "wquant", "layer", "linear",
                             "router"])
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--gemm-2sm", default="auto", choices=["0", "1", "auto"])
    ap.add_argument("--fmt", default="w8a8", choices=["w8a8", "w4a8", "w4a4"],
                    help="weight/activation formats of --kernel layer")
    args = ap.parse_args()
    dev = torch.device("cuda", 0)
    mm.set_gemm_2sm(args.gemm_2sm)
    if args.kernel == "linear":
        lshape = workloads.LINEAR_CONFIGS[args.config]
        x, w = workloads.make_linear(lshape, dev)
        lin = mm.MXFP8Linear.from_bf16(w)
        for _ in range(args.iters):
            lin(x)
        torch.cuda.synchronize()
        if mm.device_status() != 0:
            raise SystemExit("device status error")
        return
    shape = workloads.CONFIGS[args.config]
    if args.kernel == "router":
        x = workloads.make_hidden(shape, dev)
        gate = workloads.make_gate(shape, dev)
        for _ in range(args.iters):
            mm.moe_router_gate_topk(x, gate, shape.k)
        torch.cuda.synchronize()
        if mm.device_status() != 0:
            raise SystemExit("device status error")
        return
    inp = workloads.make_layer(shape, dev)
    if shape.offline:
        layer = mm.MXFP8MoELayer.from_quantized(inp["w13q"], inp["w13s"], inp["w2q"], inp["w2s"],
                                                shape.k)
    else:
        if args.kernel == "wquant":
            for _ in range(args.iters):
                mm.mx_quantize_3d(inp["w13"])
            torch.cuda.synchronize()
            return
        cls = {"w8a8": mm.MXFP8MoELayer, "w4a8": mm.W4A8MoELayer,
               "w4a4": mm.W4A4MoELayer}[args.fmt]
        if args.fmt != "w8a8" and args.kernel != "layer":
            raise SystemExit("--fmt applies to --kernel layer only")
        layer = cls.from_bf16(inp["w13"], inp["w2"], shape.k)
        del inp["w13"], inp["w2"]
    x, logits = inp["x"], inp["logits"]
    r = mm.moe_route_quant_mxfp8(x, logits, shape.k)
    aq = as_ = y = None
    if args.kernel in ("gemm2", "finalize"):
        aq, as_ = mm.grouped_gemm_swiglu_quant_mxfp8(r["xq"], r["xs"], layer.w13q, layer.w13s,
                                                     r["expert_offsets"])
    if args.kernel == "finalize":
        y = mm.grouped_gemm_mxfp8(aq, as_, layer.w2q, layer.w2s, r["expert_offsets"])
    for _ in range(args.iters):
        if args.kernel == "gemm1":
            mm.grouped_gemm_swiglu_quant_mxfp8(r["xq"], r["xs"], layer.w13q, layer.w13s,
                                               r["expert_offsets"])
        elif args.kernel == "gemm2":
            mm.grouped_gemm_mxfp8(aq, as_, layer.w2q, layer.w2s, r["expert_offsets"])
        elif args.kernel == "route":
            mm.moe_route_quant_mxfp8(x, logits, shape.k)
        elif args.kernel == "finalize":
            mm.moe_finalize_routing(y, r["topk_w"], r["src_to_sorted"], shape.k)
        elif args.kernel == "layer":
            layer(x, logits)
    torch.cuda.synchronize()
    if mm.device_status() != 0:
        raise SystemExit("device status error")


if __name__ == "__main__":
    main()
