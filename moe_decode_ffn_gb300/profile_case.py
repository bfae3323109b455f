"""A bounded decode-stack run for profilers (ncu): seeded Q4_K layers of the
Qwen3.6-35B-A3B shape (H=2048, 256 experts, top-8, I=512, Q4_K shared
expert), n_tokens tokens through n_layers layers captured as one CUDA graph
and replayed `launches` times, then the workspace status is checked.

    python -m moe_decode_ffn_gb300.profile_case --layers 4 --tokens 8 --launches 3 [--per-layer]

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
    args = ap.parse_args(argv)

    import torch

    import gen
    import moe_decode_ffn_gb300 as m

    m.build()
    spec = gen.Q4K_LAYER_SHARED_Q4_K
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
