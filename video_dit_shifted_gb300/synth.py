"""Seeded synthetic inputs.

Holds none of the method's arithmetic: it only draws i.i.d. N(0, 1) values
(torch's Philox generator on CUDA, its CPU generator otherwise) in fp32 and
casts them to the run dtype.  The same bits are copied to the host when a
check needs them, so the GPU path and any CPU check see identical inputs.
"""
import torch

# Seeds per tensor: q, k, v, text q, text k, text v, hidden rows.
SEEDS = {"q": 0, "k": 1, "v": 2, "qt": 3, "kt": 4, "vt": 5, "hidden": 6}


def normal(shape, seed, dtype=torch.bfloat16, device="cuda"):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    return x.to(dtype)


def attention_inputs(N, L, heads, head_dim, dtype=torch.bfloat16, device="cuda", base_seed=0,
                     packed=True):
    """q, k, v [N, heads, hd] and qt, kt, vt [L, heads, hd].

    With packed=True, q/k/v are views into one [N, 3, heads, hd] buffer (the
    layout a fused qkv projection produces) and so are the text tensors."""
    def draw(n, names):
        if packed:
            buf = torch.empty((n, 3, heads, head_dim), dtype=dtype, device=device)
            for i, name in enumerate(names):
                buf[:, i] = normal((n, heads, head_dim), SEEDS[name] + base_seed, dtype, device)
            return [buf[:, i] for i in range(3)], buf
        ts = [normal((n, heads, head_dim), SEEDS[name] + base_seed, dtype, device) for name in names]
        return ts, None

    (q, k, v), vid_buf = draw(N, ("q", "k", "v"))
    (qt, kt, vt), txt_buf = draw(L, ("qt", "kt", "vt"))
    return {"q": q, "k": k, "v": v, "qt": qt, "kt": kt, "vt": vt,
            "vid_buf": vid_buf, "txt_buf": txt_buf}


def hidden(N, width, dtype=torch.bfloat16, device="cuda", seed=None):
    return normal((N, width), SEEDS["hidden"] if seed is None else seed, dtype, device)
