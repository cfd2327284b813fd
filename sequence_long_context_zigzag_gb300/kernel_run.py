"""Run one kernel of the forward path a fixed number of times on prepared buffers, for an external
profiler (ncu). Nothing is printed but a one-line summary; the buffers are made before the first
profiled launch, so a profiler that counts launches sees only the setup launches and then the
kernel's.

  python -m sequence_long_context_zigzag_gb300.kernel_run --L 262144 --hq 8 --hkv 2 --ud 2 --rd 4 \
      --kernel attn --launches 2

Kernels: ``attn`` (usp_attn_fwd, FUSED ring attention), ``split_a2a`` (usp_extract_a2a of q, k, v),
``a2a_inv`` (usp_a2a4d_multi of out and lse, dir = -1), ``bwd`` (usp_attn_bwd). Inputs are N(0, 1)
bf16 drawn on the device with a seeded generator (the values play no part in what a profiler counts).
``--nseq`` packs the sequence into that many equal samples (attention only).
"""
from __future__ import annotations

import argparse

import torch

import sequence_long_context_zigzag_gb300 as usp


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--L", type=int, required=True)
    ap.add_argument("--hq", type=int, required=True)
    ap.add_argument("--hkv", type=int, required=True)
    ap.add_argument("--hd", type=int, default=128)
    ap.add_argument("--ud", type=int, required=True)
    ap.add_argument("--rd", type=int, required=True)
    ap.add_argument("--bs", type=int, default=1)
    ap.add_argument("--kernel", choices=["attn", "split_a2a", "a2a_inv", "bwd"], default="attn")
    ap.add_argument("--launches", type=int, default=1)
    ap.add_argument("--nseq", type=int, default=1)
    ap.add_argument("--noncausal", action="store_true")
    a = ap.parse_args(argv)
    if not torch.cuda.is_available():
        raise SystemExit("kernel_run needs a CUDA device")
    dev = torch.device("cuda", torch.cuda.current_device())
    bs, L, hq, hkv, hd, ud, rd = a.bs, a.L, a.hq, a.hkv, a.hd, a.ud, a.rd
    causal = not a.noncausal
    g = torch.Generator(device=dev).manual_seed(1234)
    q = torch.randn(bs, L, hq, hd, device=dev, generator=g).to(torch.bfloat16)
    k = torch.randn(bs, L, hkv, hd, device=dev, generator=g).to(torch.bfloat16)
    v = torch.randn(bs, L, hkv, hd, device=dev, generator=g).to(torch.bfloat16)
    Lr, Lu = L // rd, L // (rd * ud)
    Hkl = usp.heads_per_rank(hkv, ud)
    qh = torch.empty(rd, ud, hq // ud, bs, Lr, hd, device=dev, dtype=q.dtype)
    kh = torch.empty(rd, ud, Hkl, bs, Lr, hd, device=dev, dtype=q.dtype)
    vh = torch.empty_like(kh)
    oh = torch.empty_like(qh)
    lh = torch.empty(rd, ud, hq // ud, bs, Lr, device=dev, dtype=torch.float32)
    cu = None
    if a.nseq > 1:
        cu = torch.arange(0, L + 1, L // a.nseq, dtype=torch.int32, device=dev)
    usp.usp_extract_a2a([q, k, v], [qh, kh, vh], rd, ud)
    extra = {}
    if a.kernel in ("a2a_inv", "bwd"):
        usp.usp_attn_fwd(qh, kh, vh, oh, lh, causal=causal, hkv=hkv)
    if a.kernel == "a2a_inv":
        o_loc = torch.empty(rd, ud, bs, Lu, hq, hd, device=dev, dtype=q.dtype)
        l_loc = torch.empty(rd, ud, bs, Lu, hq, device=dev, dtype=torch.float32)
        extra = {"o_loc": o_loc, "l_loc": l_loc}
    if a.kernel == "bwd":
        dout = torch.randn(qh.shape, device=dev, generator=g).to(q.dtype)
        delta = torch.empty_like(lh)
        usp.usp_attn_bwd_delta(oh, dout, delta)
        extra = {"dout": dout, "delta": delta, "dq": torch.empty_like(qh), "dk": torch.empty_like(kh),
                 "dv": torch.empty_like(vh)}
    torch.cuda.synchronize()
    for _ in range(a.launches):
        if a.kernel == "attn":
            usp.usp_attn_fwd(qh, kh, vh, oh, lh, causal=causal, hkv=hkv, cu_seqlens=cu)
        elif a.kernel == "split_a2a":
            usp.usp_extract_a2a([q, k, v], [qh, kh, vh], rd, ud)
        elif a.kernel == "a2a_inv":
            usp.usp_a2a4d_multi([oh, lh], [extra["o_loc"], extra["l_loc"]], rd, ud, -1)
        else:
            usp.usp_attn_bwd(qh, kh, vh, extra["dout"], lh, extra["delta"], extra["dq"], extra["dk"], extra["dv"],
                             causal=causal, hkv=hkv)
    usp.usp_check()
    print(f"kernel_run: {a.launches} launch(es) of {a.kernel} at bs={bs} L={L} hq={hq} hkv={hkv} hd={hd} "
          f"u{ud}xr{rd} nseq={a.nseq}")


if __name__ == "__main__":
    main()
