"""Run one entry point of the library a few times on random inputs (for profilers and smoke runs).

    python -m exact_io_aware_07_gb300 --op fwd|gqa|splitkv|fp8|bwd --B 1 --H 32 --T 4096 --d 128 \
        [--hkv 8] [--splits 2] [--causal] [--iters 3]

Inputs are N(0, 1) (bf16, or e4m3 bytes for ``fp8``); the outputs are discarded.
The process exits non-zero if a call fails or a bounded in-kernel wait ran out.
"""
import argparse
import math


def main() -> int:
    import torch

    import exact_io_aware_07_gb300 as fa

    ap = argparse.ArgumentParser(prog="python -m exact_io_aware_07_gb300", description=__doc__,
                                 formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--op", choices=["fwd", "gqa", "splitkv", "fp8", "bwd"], default="fwd")
    ap.add_argument("--B", type=int, default=1)
    ap.add_argument("--H", type=int, default=32)
    ap.add_argument("--hkv", type=int, default=8)
    ap.add_argument("--T", type=int, default=4096)
    ap.add_argument("--d", type=int, default=128)
    ap.add_argument("--splits", type=int, default=2)
    ap.add_argument("--causal", action="store_true")
    ap.add_argument("--iters", type=int, default=3)
    a = ap.parse_args()
    fa.build()
    B, H, T, d = a.B, a.H, a.T, a.d
    scale = 1.0 / math.sqrt(d)
    g = torch.Generator(device="cuda").manual_seed(0)

    def rnd(*shape):
        return torch.randn(*shape, device="cuda", generator=g).to(torch.bfloat16)

    q = rnd(B, H, T, d)
    kv_heads = a.hkv if a.op == "gqa" else H
    k, v = rnd(B, kv_heads, T, d), rnd(B, kv_heads, T, d)
    o = torch.empty(B, H, T, d, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, H, T, dtype=torch.float32, device="cuda")
    if a.op == "splitkv":
        ws = torch.empty(fa.fa_fwd_splitkv_workspace_bytes(B, H, T, d, a.splits), dtype=torch.uint8, device="cuda")
    elif a.op == "fp8":
        ws = torch.empty(fa.fa_fwd_fp8_workspace_bytes(B, H, T, d), dtype=torch.uint8, device="cuda")
        q8, k8, v8 = (t.float().to(torch.float8_e4m3fn).view(torch.uint8) for t in (q, k, v))
    elif a.op == "bwd":
        fa.fa_fwd(q, k, v, o, lse, a.causal, scale)
        do = rnd(B, H, T, d)
        dq, dk, dv = (torch.empty_like(q) for _ in range(3))
        ws = torch.empty(fa.fa_bwd_workspace_bytes(B, H, T), dtype=torch.uint8, device="cuda")
    for _ in range(a.iters):
        if a.op == "fwd":
            fa.fa_fwd(q, k, v, o, lse, a.causal, scale)
        elif a.op == "gqa":
            fa.fa_fwd_gqa(q, k, v, o, lse, a.causal, scale)
        elif a.op == "splitkv":
            fa.fa_fwd_splitkv(q, k, v, o, lse, a.causal, scale, a.splits, ws)
        elif a.op == "fp8":
            fa.fa_fwd_fp8(q8, k8, v8, o, lse, a.causal, scale, (1.0, 1.0, 1.0), ws)
        else:
            fa.fa_bwd(q, k, v, o, lse, do, dq, dk, dv, a.causal, scale, ws)
    torch.cuda.synchronize()
    status = fa.fa_device_status()
    print(f"{a.op}: {a.iters} calls, B={B} H={H} T={T} d={d} causal={a.causal}, device status {status}")
    return 0 if status == 0 else 1


if __name__ == "__main__":
    raise SystemExit(main())
