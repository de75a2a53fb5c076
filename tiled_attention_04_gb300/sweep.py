"""Latency sweep of these kernels against plain PyTorch ("vanilla") attention.

The field guide's "Systems and Parallelism" §1.3 asks for a flash_benchmarking
table: forward, backward and end-to-end (forward plus backward) latency of the
flash kernel and of the regular PyTorch attention, over sequence lengths,
head dimensions and precisions, batch 1 and causal masking, with out-of-memory
cells reported as results.  The grid below is this module's choice (the
pages' own values did not survive): N = 128 ... 32768 in powers of two,
d in {16, 32, 64, 128}, bf16 and fp32.

Vanilla attention is the textbook form in PyTorch operations, materialising
the score matrix: S = scale * Q K^T, masked with -inf above the diagonal,
P = softmax(S) in fp32, O = P V, with autograd for the backward pass.  The
flash side is the C-ABI path (fa_fwd, then fa_bwd with a workspace allocated
outside the timed region).

Timing: CUDA events on the current stream around each call, after warm-up;
the L2 cache (129 MB) is flushed before every timed call by writing a 256 MiB
buffer; the median of `reps` calls is reported, in milliseconds.

fp32 cells run in the library's fp32 mode (--fp32-mode; default auto: split
bf16 pairs on the tensor cores for d <= 64 at this scale, see include/fa.h).

Run: python -m tiled_attention_04_gb300.sweep [--reps R] [--max-n N] [--json PATH] [--fp32-mode M]
     python -m tiled_attention_04_gb300.sweep --layer [--non-causal]   (the xl attention block)
"""
from __future__ import annotations

import argparse
import json
import math
import sys

SEQ = [128 << i for i in range(9)]       # 128 ... 32768
DIMS = [16, 32, 64, 128]
DTYPES = ["bf16", "fp32"]


def _torch():
    import torch
    return torch


def vanilla(Q, K, V, causal, scale):
    """Attention with the score matrix materialised (softmax in fp32 or wider)."""
    torch = _torch()
    S = torch.matmul(Q, K.transpose(-1, -2))
    S = (S.float() if S.element_size() < 4 else S) * scale
    if causal:
        n_q, n_k = S.shape[-2], S.shape[-1]
        mask = torch.ones(n_q, n_k, dtype=torch.bool, device=S.device).triu(1)
        S = S.masked_fill(mask, float("-inf"))
    P = torch.softmax(S, dim=-1).to(V.dtype)
    return torch.matmul(P, V)


class Timer:
    def __init__(self, reps, warmup):
        torch = _torch()
        self.reps, self.warmup = reps, warmup
        self.flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")

    def __call__(self, fn, setup=None):
        """Median milliseconds of fn(); setup() (untimed) runs before each call."""
        torch = _torch()
        times = []
        for i in range(self.warmup + self.reps):
            if setup is not None:
                setup()
            self.flush.zero_()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            b.synchronize()
            if i >= self.warmup:
                times.append(a.elapsed_time(b))
        times.sort()
        return times[len(times) // 2]


def measure_cell(N, d, dtype, causal, timer):
    """{'flash': (fwd, bwd, e2e), 'vanilla': (fwd, bwd, e2e) or 'OOM'} in ms."""
    torch = _torch()
    from . import binding
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    g = torch.Generator(device="cuda")
    g.manual_seed(N * 1000 + d)
    Q, K, V, dO = (torch.randn(1, 1, N, d, generator=g, device="cuda", dtype=torch.float32).to(tdt)
                   for _ in range(4))
    scale = 1.0 / math.sqrt(d)
    out = {}

    # ---- flash (C ABI)
    ws = binding.alloc_workspace(Q, K, causal)
    O, L = binding.fa_fwd(Q, K, V, is_causal=causal)
    dQ, dK, dV = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)
    f_fwd = timer(lambda: binding.fa_fwd(Q, K, V, is_causal=causal, O=O, L=L))
    f_bwd = timer(lambda: binding.fa_bwd(Q, K, V, O, dO, L, is_causal=causal, dQ=dQ, dK=dK, dV=dV, workspace=ws))

    def flash_e2e():
        binding.fa_fwd(Q, K, V, is_causal=causal, O=O, L=L)
        binding.fa_bwd(Q, K, V, O, dO, L, is_causal=causal, dQ=dQ, dK=dK, dV=dV, workspace=ws)
    out["flash"] = (f_fwd, f_bwd, timer(flash_e2e))
    del ws, O, L, dQ, dK, dV

    # ---- vanilla (PyTorch operations, autograd backward)
    try:
        q, k, v = (t.clone().requires_grad_(True) for t in (Q, K, V))
        with torch.no_grad():
            v_fwd = timer(lambda: vanilla(Q, K, V, causal, scale))
        state = {}

        def fwd_for_bwd():
            state["o"] = vanilla(q, k, v, causal, scale)

        def bwd():
            state["o"].backward(dO)
        v_bwd = timer(bwd, setup=fwd_for_bwd)

        def vanilla_e2e():
            vanilla(q, k, v, causal, scale).backward(dO)
        out["vanilla"] = (v_fwd, v_bwd, timer(vanilla_e2e))
        del state, q, k, v
    except torch.cuda.OutOfMemoryError:
        out["vanilla"] = "OOM"
    torch.cuda.empty_cache()
    return out


def layer_block(B=4, N=1024, H=25, d=64, causal=True, reps=20, warmup=5):
    """Milliseconds of one forward plus backward pass of an attention block of the
    xl model's shape (d_model 1600 = 25 heads of 64; the field guide's "Model
    configurations"): fused QKV projection, attention, output projection, in
    bf16 with random-init weights, for three attention functions -- these
    kernels (through patch_sdpa), PyTorch's own scaled_dot_product_attention,
    and the vanilla form above."""
    torch = _torch()
    import torch.nn.functional as F
    from .autograd import patch_sdpa
    D = H * d
    g = torch.Generator(device="cuda")
    g.manual_seed(1600)
    x = torch.randn(B, N, D, generator=g, device="cuda").to(torch.bfloat16).requires_grad_(True)
    bound = math.sqrt(6.0 / (D + 3 * D))
    w_qkv = ((torch.rand(D, 3 * D, generator=g, device="cuda") * 2 - 1) * bound).to(torch.bfloat16)
    w_o = ((torch.rand(D, D, generator=g, device="cuda") * 2 - 1) * math.sqrt(3.0 / D)).to(torch.bfloat16)
    w_qkv.requires_grad_(True)
    w_o.requires_grad_(True)
    grad = torch.randn(B, N, D, generator=g, device="cuda").to(torch.bfloat16)

    def block(attn):
        qkv = (x @ w_qkv).view(B, N, 3, H, d)
        q, k, v = (qkv[:, :, i].transpose(1, 2) for i in range(3))
        o = attn(q, k, v)
        (o.transpose(1, 2).reshape(B, N, D) @ w_o).backward(grad)

    timer = Timer(reps, warmup)
    out = {}
    with patch_sdpa():
        out["flash"] = timer(lambda: block(lambda q, k, v: F.scaled_dot_product_attention(q, k, v,
                                                                                          is_causal=causal)))
    out["torch_sdpa"] = timer(lambda: block(lambda q, k, v: F.scaled_dot_product_attention(q, k, v,
                                                                                           is_causal=causal)))
    out["vanilla"] = timer(lambda: block(lambda q, k, v: vanilla(q, k, v, causal, 1.0 / math.sqrt(d))))
    return out


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--reps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--max-n", type=int, default=SEQ[-1])
    ap.add_argument("--dims", default=",".join(map(str, DIMS)))
    ap.add_argument("--dtypes", default=",".join(DTYPES))
    ap.add_argument("--non-causal", action="store_true")
    ap.add_argument("--json", default=None, help="also write the cells as JSON lines to this file")
    ap.add_argument("--layer", action="store_true", help="time the xl-shaped attention block instead")
    ap.add_argument("--fp32-mode", choices=("auto", "exact", "split"), default="auto",
                    help="the library's fp32 mode for the fp32 cells")
    a = ap.parse_args(argv)
    torch = _torch()
    if not torch.cuda.is_available():
        raise SystemExit("the sweep needs a CUDA device")
    from . import binding
    binding.set_fp32_mode({"auto": binding.FA_FP32_AUTO, "exact": binding.FA_FP32_EXACT,
                           "split": binding.FA_FP32_SPLIT}[a.fp32_mode])
    causal = not a.non_causal
    if a.layer:
        res = layer_block(causal=causal)
        print(json.dumps({"block": "xl attention (B 4, N 1024, d_model 1600, 25 heads), fwd+bwd, bf16",
                          "causal": causal, "unit": "ms", **{k: round(v, 4) for k, v in res.items()}}))
        return res
    timer = Timer(a.reps, a.warmup)
    rows = []
    fh = open(a.json, "w") if a.json else None
    print("| dtype | d | N | flash fwd | flash bwd | flash e2e | vanilla fwd | vanilla bwd | vanilla e2e | e2e speed-up |")
    print("|---|---|---|---|---|---|---|---|---|---|")
    for dt in a.dtypes.split(","):
        for d in map(int, a.dims.split(",")):
            for N in (n for n in SEQ if n <= a.max_n):
                cell = measure_cell(N, d, dt, causal, timer)
                f = cell["flash"]
                v = cell["vanilla"]
                if v == "OOM":
                    vcols, sp = "OOM | OOM | OOM", "-"
                else:
                    vcols = " | ".join(f"{x:.3f}" for x in v)
                    sp = f"{v[2] / f[2]:.1f}x"
                print(f"| {dt} | {d} | {N} | {f[0]:.3f} | {f[1]:.3f} | {f[2]:.3f} | {vcols} | {sp} |")
                sys.stdout.flush()
                rec = {"dtype": dt, "d": d, "N": N, "causal": causal, "batch": 1, "heads": 1, "unit": "ms",
                       "fp32_mode": a.fp32_mode if dt == "fp32" else None,
                       "flash": {"fwd": f[0], "bwd": f[1], "e2e": f[2]},
                       "vanilla": v if v == "OOM" else {"fwd": v[0], "bwd": v[1], "e2e": v[2]}}
                rows.append(rec)
                if fh:
                    fh.write(json.dumps(rec) + "\n")
                    fh.flush()
    if fh:
        fh.close()
    return rows


if __name__ == "__main__":
    main()
