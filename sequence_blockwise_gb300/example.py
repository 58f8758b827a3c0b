"""Example of the Python binding: two packed documents with causal masks, the
TASP schedule over 8 virtual sequence-parallel ranks, the forward and the
backward on one GPU. Run with `python -m sequence_blockwise_gb300.example`."""
import torch

import sequence_blockwise_gb300 as sb


def run(seed: int = 0):
    torch.manual_seed(seed)
    cu = [0, 1000, 4096]                                       # two packed documents
    q = torch.randn(4096, 32, 128, device="cuda").bfloat16()   # [T, Hq, d]
    k = torch.randn(4096, 8, 128, device="cuda").bfloat16()    # [T, Hkv, d]
    v = torch.randn_like(k)

    att = sb.PackedAttention(cu, causal=True, kind=sb.SP_SCHED_TASP, P=8, Hq=32)
    o, lse = att(q, k, v)                 # o [T, Hq, d] bf16, lse [Hq, T] fp32 (natural log)
    dq, dk, dv = att.backward(q, k, v, o, lse, torch.randn_like(q))
    return dict(cu=cu, q=q, k=k, v=v, o=o, lse=lse, dq=dq, dk=dk, dv=dv)


if __name__ == "__main__":
    out = run()
    for name in ("o", "lse", "dq", "dk", "dv"):
        print(f"{name}: {tuple(out[name].shape)} {out[name].dtype}")
