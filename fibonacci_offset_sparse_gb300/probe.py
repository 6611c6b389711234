"""Synthetic retrieval probe of learned-alpha dynamics.

The pages report that a learned dilation stays near its initial value ("Depth-Staggered
Fibonacci Spacing for Sparse Attention", Key results: learned dilation is inert); their task
data are not available, so this probe defines its own synthetic task.  One layer, INTERP
mode, alpha = 1 + 0.5 tanh(theta) learned by gradient descent on theta through the library's
backward (dl/dalpha).

Task: key rows k_j ~ N(0, I); query i is built so that, after RoPE at the rows' own
positions, it matches key i - d* exactly (q'_i = k'_{i-d*}, score |k|^2/8 ~ 8) and no other
key beyond chance (scores ~ N(0, 1)); values v_j ~ N(0, I); the loss is the mean of
|O_i - v_{i-d*}|^2 over the queries i >= d*.  The key at distance d* is attended only when a
rung lands within one row of it (the interpolated rows of rung f are floor(alpha f) and the
row before), so a rung more than one row away gives no gradient toward it.

    python -m fibonacci_offset_sparse_gb300.probe --targets 30 35 --steps 200

prints one JSON line per target with the alpha and loss trajectories.
"""
import argparse
import json

import numpy as np
import torch

from . import fib_attn as fa
from . import inputs
from .autograd import fib_attention

PROBE_CONFIG = 40  # seed stream of the probe's inputs


def rotate(x: np.ndarray, angle_per_freq: np.ndarray) -> np.ndarray:
    """Rotate-half pairs (m, m + D/2) of x[..., D] by angle_per_freq[..., D/2] (float64)."""
    h = x.shape[-1] // 2
    c, s = np.cos(angle_per_freq), np.sin(angle_per_freq)
    a, b = x[..., :h], x[..., h:]
    return np.concatenate([a * c - b * s, a * s + b * c], axis=-1)


def make_task(B: int, H: int, N: int, target: int, rope_base: float = 10000.0, seed: int = inputs.SEED):
    """(q, k, v, target values) float32 CPU tensors [B, H, N, 64] of the retrieval task."""
    D = 64
    draw = lambda shape, tid: inputs.normal(shape, PROBE_CONFIG, target, tid, "f32", seed).double().numpy()
    k = draw((B, H, N, D), inputs.TENSOR_K)
    v = draw((B, H, N, D), inputs.TENSOR_V)
    theta = rope_base ** (-2.0 * np.arange(D // 2) / D)
    q = np.zeros_like(k)
    # q_i = R(-d*) k_{i-d*}: then R(i) q_i = R(i - d*) k_{i-d*}, the key's own rotated row
    q[:, :, target:] = rotate(k[:, :, : N - target], (-target * theta)[None, None, None, :])
    q[:, :, :target] = draw((B, H, target, D), inputs.TENSOR_Q)
    y = np.zeros_like(v)
    y[:, :, target:] = v[:, :, : N - target]
    f = lambda a: torch.from_numpy(a.astype(np.float32))
    return f(q), f(k), f(v), f(y)


def run(target: int, steps: int = 200, lr: float = 1e-3, B: int = 4, H: int = 2, N: int = 512, W: int = 12,
        dtype=torch.float32, device: str = "cuda", record_every: int = 10):
    """Gradient descent on theta (alpha = 1 + 0.5 tanh theta, theta_0 = 0) for one target."""
    plan = fa.fib_attn_plan_create(fa.FIB_BASE_FIBONACCI, [1.0], W, N, fa.FIB_MODE_INTERP)
    q, k, v, y = (t.to(device=device, dtype=dtype) for t in make_task(B, H, N, target))
    y = y.float()
    theta = torch.zeros(1, dtype=torch.float32, device=device, requires_grad=True)
    opt = torch.optim.SGD([theta], lr=lr)
    hist = {"step": [], "alpha": [], "loss": [], "dalpha": []}
    for step in range(steps + 1):
        alpha = 1.0 + 0.5 * torch.tanh(theta)
        alpha_leaf = alpha.detach().clone().requires_grad_(True)
        o = fib_attention(plan, 0, q, k, v, alpha_leaf)
        loss = ((o.float() - y)[:, :, target:] ** 2).mean()
        loss.backward()
        da = float(alpha_leaf.grad[0])
        if step % record_every == 0 or step == steps:
            hist["step"].append(step)
            hist["alpha"].append(float(alpha.detach()[0]))
            hist["loss"].append(float(loss.detach()))
            hist["dalpha"].append(da)
        if step == steps:
            break
        opt.zero_grad()
        alpha.backward(alpha_leaf.grad)  # chain rule to theta
        opt.step()
    plan.close()
    rungs = [f for f in fa.fib_attn_base(fa.FIB_BASE_FIBONACCI) if f > W - 1]
    nearest = min(rungs, key=lambda f: abs(f - target))
    return {"target": target, "steps": steps, "lr": lr, "shape": [B, H, N, 64], "W": W,
            "dtype": str(dtype).replace("torch.", ""), "nearest_rung_at_alpha_1": nearest,
            "rows_from_target_at_alpha_1": nearest - target, **hist}


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--targets", type=int, nargs="+", default=[30, 34, 35])
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--lr", type=float, default=1e-3)
    ap.add_argument("--bf16", action="store_true")
    args = ap.parse_args()
    fa.lib()
    for tg in args.targets:
        r = run(tg, args.steps, args.lr, dtype=torch.bfloat16 if args.bf16 else torch.float32)
        print(json.dumps(r))


if __name__ == "__main__":
    main()
