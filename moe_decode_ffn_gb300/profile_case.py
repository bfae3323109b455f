"""A bounded decode-stack run for profilers (ncu): seeded Q4_K layers of the
Qwen3.6-35B-A3B shape (H=2048, 256 experts, top-8, I=512, Q4_K shared
expert), n_tokens tokens through n_layers layers captured as one CUDA graph
and replayed `launches` times, then the workspace status is checked.

    python -m moe_decode_ffn_gb300.profile_case --layers 4 --tokens 8 --launches 3 [--per-layer]
    python -m moe_decode_ffn_gb300.profile_case --spec bf16 --layers 4 --tokens 2 --launches 2
    python -m moe_decode_ffn_gb300.profile_case --batched 64 --mode tensor --launches 3

The last form runs the batched routed FFN of one Qwen3-30B-A3B-shaped layer
(128 experts, I=768, no shared expert, Q4_K) for T tokens with per-token
routing, in the integer (int8) or tensor-core (tensor) mode.

`--spec bf16` takes the bf16 layer of the same shape (bf16 routed and shared
experts, four kernels per layer) instead of the all-Q4_K one.

It exits non-zero if the device recorded an error, so a profiler is only ever
run on a command that has just exited 0 on its own.
"""
from __future__ import annotations

import argparse
import sys


def main(argv=None) -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--layers", type=int, default=4)
    ap.add_argument("--tokens", type=int, default=8)
    ap.add_argument("--launches", type=int, default=3)
    ap.add_argument("--seed", type=int, default=21)
    ap.add_argument("--per-layer", action="store_true", help="four kernels per layer instead of "
                    "the persistent kernel")
    ap.add_argument("--batched", type=int, default=0, help="T: batched FFN of T tokens instead")
    ap.add_argument("--mode", default="tensor", choices=["tensor", "int8"])
    ap.add_argument("--spec", default="q4k", choices=["q4k", "bf16"])
    args = ap.parse_args(argv)

    import torch

    import gen
    import moe_decode_ffn_gb300 as m

    m.build()
    if args.batched:
        T = args.batched
        L = m.device_layer(gen.Q4K_LAYER_128E, args.seed, 0)
        x = gen.make_tokens(args.seed + 1, T, device="cuda")
        keys = gen.raw64([gen.stream_key(args.seed, t, 901) for t in range(T)], 128)
        ids = torch.argsort(keys, dim=1)[:, :8].to(torch.int32).cuda()
        w = torch.full((T, 8), 0.125, dtype=torch.float32, device="cuda")
        mode = m.SI_FFN_TENSOR if args.mode == "tensor" else m.SI_FFN_INT8
        ws = m.workspace(m.ffn_batched_workspace_bytes(L, T))
        for _ in range(args.launches):
            m.si_moe_ffn_batched(L, x, ids, w, mode, ws=ws)
        torch.cuda.synchronize()
        st = m.si_workspace_status(ws)
        print(f"batched T={T} mode={args.mode} launches={args.launches} status={m.status_string(st)}")
        return 0 if st == m.SI_OK else 1
    spec = gen.BF16_LAYER if args.spec == "bf16" else gen.Q4K_LAYER_SHARED_Q4_K
    layers = [m.device_layer(spec, args.seed, l) for l in range(args.layers)]
    x = gen.make_tokens(args.seed + 1, args.tokens, device="cuda")
    mode = m.SI_STACK_PER_LAYER if args.per_layer else m.SI_STACK_AUTO
    g = m.StackGraph(layers, x, mode=mode)
    for _ in range(args.launches):
        g.launch()
    torch.cuda.synchronize()
    st = m.si_workspace_status(g.ws)
    print(f"layers={args.layers} tokens={args.tokens} launches={args.launches} "
          f"persistent={g.persistent} status={m.status_string(st)}")
    g.close()
    return 0 if st == m.SI_OK else 1


if __name__ == "__main__":
    sys.exit(main())
