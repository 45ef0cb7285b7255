"""Seeded synthetic inputs for the MoE block (shared by the tests, the benchmark
and the smoke check; imported by both the CUDA-path callers and the oracle
callers, and holding none of the block's arithmetic).

Recipe: a seeded torch.Generator on the target device draws, in this order,
x ~ N(0,1) [T,H], W_router ~ N(0, 0.02^2) [E,H], W_gate and W_up
~ N(0, 0.02^2) [E,I,H], W_down ~ N(0, 0.02^2) [E,H,I]; each is drawn in fp32
and rounded to bf16.  Shapes follow the Qwen3-235B-A22B config quoted on the
csdn page "MoE架构深度解析：128专家与8激活的智能路由" (128 experts, 8 per token,
moe_intermediate_size 1536, hidden 4096) and smaller layers of the same form.

Skewed routing: the router has no bias term, so a per-expert bias is carried
in-band: x[:,0] = 1 and W_router[e,0] = b_e.  b is calibrated here on a
statistical model of the logits (b_e plus i.i.d. N(0, sigma^2) noise with
sigma = 0.02*sqrt(H-1), the spread of the remaining x·W terms) so that the
share of token-expert pairs each expert receives follows Zipf(s) over a seeded
permutation of the experts, water-filled at 0.999/K (top-K with distinct
experts cannot give any expert more than 1/K of the pairs).  The calibration
samples synthetic noise, never the router.
"""
from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int
    H: int
    E: int
    K: int
    I: int
    norm: bool
    zipf: float = 0.0  # > 0: skewed routing with this Zipf exponent
    seed: int = 0
    note: str = field(default="", compare=False)

    @property
    def pairs(self):
        return self.T * self.K


CONFIGS = {
    "tiny": MoEConfig("tiny", 64, 128, 8, 2, 256, False,
                      note="T=64 H=128 E=8 K=2 I=256 norm_topk_prob=false"),
    "prefill_h2048": MoEConfig("prefill_h2048", 4096, 2048, 128, 8, 768, True,
                               note="Qwen3-style prefill layer T=4096 H=2048 E=128 K=8 I=768"),
    "prefill_h4096": MoEConfig("prefill_h4096", 8192, 4096, 128, 8, 1536, True,
                               note="large-expert prefill T=8192 H=4096 E=128 K=8 I=1536"),
    "decode_t1": MoEConfig("decode_t1", 1, 4096, 128, 8, 1536, True),
    "decode_t4": MoEConfig("decode_t4", 4, 4096, 128, 8, 1536, True),
    "decode_t16": MoEConfig("decode_t16", 16, 4096, 128, 8, 1536, True),
    "decode_t64": MoEConfig("decode_t64", 64, 4096, 128, 8, 1536, True),
    "skew": MoEConfig("skew", 16384, 4096, 128, 8, 1536, True, zipf=1.2,
                      note="T=16384 H=4096 E=128 K=8 I=1536, Zipf(1.2) expert popularity"),
    # few big experts, top-2 without renormalisation (the Mixtral-style router
    # the cnblogs page contrasts with norm_topk_prob); H and I of a 4096-wide
    # model with 3.5x wide experts
    "mixtral_prefill": MoEConfig("mixtral_prefill", 4096, 4096, 8, 2, 14336, False,
                                 note="T=4096 H=4096 E=8 K=2 I=14336 norm_topk_prob=false"),
    "mixtral_decode_t1": MoEConfig("mixtral_decode_t1", 1, 4096, 8, 2, 14336, False,
                                   note="T=1 H=4096 E=8 K=2 I=14336 norm_topk_prob=false"),
}


def zipf_targets(E, K, s, seed=0, cap_frac=0.999):
    """Target pair share per expert: Zipf(s) over ranks of a seeded expert
    permutation, water-filled so that no share exceeds cap_frac/K."""
    ranks = np.arange(1, E + 1, dtype=np.float64)
    q = ranks ** (-s)
    q /= q.sum()
    cap = cap_frac / K
    fixed = np.zeros(E, bool)
    for _ in range(E):
        over = (q > cap) & ~fixed
        if not over.any():
            break
        fixed |= over
        q[fixed] = cap
        free = ~fixed
        q[free] *= (1.0 - cap * fixed.sum()) / q[free].sum()
    perm = np.random.default_rng(seed + 7919).permutation(E)
    target = np.empty(E)
    target[perm] = q  # expert perm[r] gets the share of rank r+1
    return target


def zipf_bias(E, K, H, s, seed=0, samples=20000, iters=60):
    """Per-expert logit offsets b (float64 [E]) that realise zipf_targets
    under the noise model described in the module docstring."""
    target = zipf_targets(E, K, s, seed)
    sigma = 0.02 * np.sqrt(H - 1)
    rng = np.random.default_rng(seed + 104729)
    noise = rng.standard_normal((samples, E)) * sigma
    b = sigma * np.log(target * E)
    floor = 0.5 / (samples * K)
    for _ in range(iters):
        z = noise + b
        top = np.argpartition(-z, K - 1, axis=1)[:, :K]
        obs = np.bincount(top.ravel(), minlength=E) / (samples * K)
        b += 0.5 * sigma * (np.log(target) - np.log(np.maximum(obs, floor)))
        b -= b.mean()
    return b, target


def make_inputs(cfg: MoEConfig, device="cpu", seed=None):
    """Draw the block inputs for cfg.  Returns a dict of bf16 tensors on device:
    x [T,H], W_router [E,H], W_gate [E,I,H], W_up [E,I,H], W_down [E,H,I]."""
    seed = cfg.seed if seed is None else seed
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(seed)

    def draw(shape, std):
        t = torch.randn(shape, generator=g, device=dev, dtype=torch.float32)
        if std != 1.0:
            t.mul_(std)
        return t.to(torch.bfloat16)

    T, H, E, I = cfg.T, cfg.H, cfg.E, cfg.I
    x = draw((T, H), 1.0)
    Wr = draw((E, H), 0.02)
    Wg = draw((E, I, H), 0.02)
    Wu = draw((E, I, H), 0.02)
    Wd = draw((E, H, I), 0.02)
    if cfg.zipf > 0:
        b, _ = zipf_bias(E, cfg.K, H, cfg.zipf, seed)
        x[:, 0] = 1.0
        Wr[:, 0] = torch.tensor(b, dtype=torch.float32).to(torch.bfloat16).to(dev)
    return dict(x=x, W_router=Wr, W_gate=Wg, W_up=Wu, W_down=Wd)


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> host numpy uint16 array of its bit patterns."""
    assert t.dtype == torch.bfloat16
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def from_bits(a: np.ndarray, device="cpu") -> torch.Tensor:
    """numpy uint16 bit patterns -> bf16 tensor."""
    return torch.from_numpy(np.ascontiguousarray(a, np.uint16).view(np.int16)).view(
        torch.bfloat16).to(device)


def sample_rows(T, n, seed=0):
    """A seeded, sorted sample of n distinct token rows (always includes the
    first and last token, so ragged tails are covered)."""
    if n >= T:
        return np.arange(T, dtype=np.int32)
    rng = np.random.default_rng(seed + 31337)
    pick = rng.choice(np.arange(1, T - 1), size=max(n - 2, 0), replace=False)
    return np.sort(np.concatenate([[0, T - 1], pick])).astype(np.int32)
