"""Seeded synthetic workloads for the draft-block select-and-verify step.

This module draws inputs only. It holds none of the step's arithmetic (no
top-K, pair scores, path search or verification). The same generator feeds
the CUDA path and the fp64 oracle, so both see identical bytes.

The workloads follow the shapes of the DFlash 2 pages: block sizes 4 to 16,
K = 16 candidates, a Qwen-family vocabulary of 151936 and drafter widths
4096/5120. No trained drafter, target model or dataset is involved.

Recipe, for every workload:
  * hidden states h ~ N(0, 1), shape [B, L, d]. Row 0 of each block is the
    verified slot; rows 1..L-1 are the draft positions.
  * LM head W_vocab ~ N(0, 1/d), shape [d, V]. Gate W_g ~ N(0, 1/d), shape
    [r, d]. Selector tables A, B ~ N(0, 1/r), shape [V, r].
  * last verified token x0 ~ U{0..V-1}, one per request.
  * Zipf-shaped rows (the throughput workload): add off_v = -1.1 ln(pi(v)+1),
    with pi a seeded permutation of the vocabulary. The offset is folded into
    the product, so the boundary stays bias-free: h[..., d-1] = 8 and
    W[d-1, v] = off_v / 8.
  * everything is rounded to the workload dtype (bf16, or fp32 for the tiny
    case) before anything is derived from it.
  * target logits Z [B, L, V]: row i is the target's prediction after x_i.
    Z[b, i] = u[b, i+1] + sigma_{i+1} * n (i < L-1), Z[b, L-1] = u[b, L-1] +
    sigma_{L-1} * n', with u a reference product h . W computed here with a
    torch library matmul. That product exists only to correlate the synthetic
    target with the drafter. Neither the oracle nor the CUDA path reads it:
    both recompute their own logits from h and W. sigma is bisected on
    separate calibration noise to hit the agreement the workload asks for:
    top-1 agreement (argmax Z row == drafter argmax), or recall@16 (argmax Z
    row lies in the drafter's top 16), per position where the rate varies.
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class WorkloadSpec:
    name: str
    B: int
    L: int
    V: int
    d: int
    r: int
    dtype: str = "bf16"  # "bf16" or "fp32"
    seed: int = 0
    K: int = 16
    # target agreement: ("top1", rate) | ("recall16", rate) | ("top1_linear", first, last)
    agreement: tuple = ("top1", 0.85)
    zipf: bool = False
    # "e4m3": the LM head is also given quantised, Wq [V, d] E4M3 bytes with one power-of-two
    # scale per vocabulary entry, drawn from the same W
    lmhead: str = "bf16"
    path_modes: tuple = ("viterbi",)
    temperatures: tuple = (0.0,)

    @property
    def rows(self) -> int:
        return self.B * self.L

    def with_(self, **kw) -> "WorkloadSpec":
        return dataclasses.replace(self, **kw)


# The five workloads of the pages' draft-block step (block 8 is the serving default,
# block 16 the long-block case, the tiny one is checkable by brute force).
TINY = WorkloadSpec("tiny_B1_L4_V1024_d256_r32_fp32", B=1, L=4, V=1024, d=256, r=32,
                    dtype="fp32", seed=0, agreement=("top1", 0.85), path_modes=("viterbi",),
                    temperatures=(0.0,))
SINGLE = WorkloadSpec("single_B1_L8_V151936_d5120", B=1, L=8, V=151936, d=5120, r=256,
                      seed=1, agreement=("top1", 0.85), path_modes=("viterbi",),
                      temperatures=(0.0,))
SMALL_BATCH = WorkloadSpec("small_batch_B8_L8_V151936_d5120", B=8, L=8, V=151936, d=5120,
                           r=256, seed=2, agreement=("recall16", 0.99), path_modes=("greedy",),
                           temperatures=(1.0,))
THROUGHPUT = WorkloadSpec("throughput_B32_L8_V151936_d5120_zipf", B=32, L=8, V=151936, d=5120,
                          r=256, seed=3, agreement=("top1", 0.85), zipf=True,
                          path_modes=("greedy", "viterbi"), temperatures=(0.0, 0.6))
LONG_BLOCK = WorkloadSpec("long_block_B16_L16_V151936_d4096", B=16, L=16, V=151936, d=4096,
                          r=256, seed=4, agreement=("top1_linear", 0.85, 0.55),
                          path_modes=("viterbi", "greedy"), temperatures=(0.0, 1.0))

# The throughput workload with a 65536-token vocabulary: the same per-tile work and several
# tiles per SM, W_vocab (671 MB) still five times L2, small enough for multi-pass profiler
# captures.
THROUGHPUT_PROFILE = THROUGHPUT.with_(name="throughput_B32_L8_V65536_d5120_zipf", V=65536)

# The throughput workload with blocks of 9: 288 rows, of which 256 are drafted, so skipping the
# verified slots saves a whole pass over W_vocab (the vocabulary-major LM head).
THROUGHPUT_BLOCK9 = THROUGHPUT.with_(name="throughput_B32_L9_V151936_d5120_zipf", L=9)

WORKLOADS = {w.name: w for w in (TINY, SINGLE, SMALL_BATCH, THROUGHPUT, LONG_BLOCK,
                                 THROUGHPUT_PROFILE, THROUGHPUT_BLOCK9)}


def torch_dtype(spec: WorkloadSpec) -> torch.dtype:
    return torch.bfloat16 if spec.dtype == "bf16" else torch.float32


def _reference_product(h: torch.Tensor, W: torch.Tensor, chunk: int = 32768) -> torch.Tensor:
    """fp32 library product h[B, L-1, d] @ W[d, V] -> [B, L-1, V] (input synthesis only)."""
    B, P, d = h.shape
    V = W.shape[1]
    hf = h.reshape(B * P, d).float()
    out = torch.empty(B * P, V, dtype=torch.float32, device=h.device)
    for v0 in range(0, V, chunk):
        out[:, v0:v0 + chunk] = hf @ W[:, v0:v0 + chunk].float()
    return out.reshape(B, P, V)


def _rate(u: torch.Tensor, sigma: float, noise: torch.Tensor, kind: str) -> float:
    """Agreement of argmax(u + sigma*noise) with the drafter: u [n, V], noise [R, n, V]."""
    y = (u.unsqueeze(0) + sigma * noise).argmax(-1)  # [R, n]
    if kind == "top1":
        return (y == u.argmax(-1).unsqueeze(0)).float().mean().item()
    top = u.topk(16, dim=-1).indices  # [n, 16]
    return (y.unsqueeze(-1) == top.unsqueeze(0)).any(-1).float().mean().item()


def _bisect_sigma(u: torch.Tensor, target: float, kind: str, gen: torch.Generator,
                  reps: int | None, iters: int = 22) -> float:
    if reps is None:
        reps = max(2, min(512, (1 << 25) // max(1, u.numel())))
    noise = torch.randn((reps,) + tuple(u.shape), generator=gen, device=u.device)
    lo, hi = 0.0, 8.0 * float(u.std().item()) + 1e-6
    for _ in range(iters):
        mid = 0.5 * (lo + hi)
        if _rate(u, mid, noise, kind) > target:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


def generate(spec: WorkloadSpec, device="cpu", *, calib_reps: int | None = None) -> dict:
    """Draw one workload on `device`. Returns a dict of tensors (h, W, Wg, A, Bt, x0, Z)
    plus 'meta' (noise scales and the agreement actually realised)."""
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(spec.seed)
    B, L, V, d, r = spec.B, spec.L, spec.V, spec.d, spec.r
    if L < 2 or V < spec.K:
        raise ValueError("a workload needs L >= 2 and V >= K")
    dt = torch_dtype(spec)

    h = torch.randn(B, L, d, generator=gen, device=device)
    W = torch.randn(d, V, generator=gen, device=device) / math.sqrt(d)
    Wg = torch.randn(r, d, generator=gen, device=device) / math.sqrt(d)
    A = torch.randn(V, r, generator=gen, device=device) / math.sqrt(r)
    Bt = torch.randn(V, r, generator=gen, device=device) / math.sqrt(r)
    x0 = torch.randint(0, V, (B,), generator=gen, device=device, dtype=torch.int64)
    if spec.zipf:
        perm = torch.randperm(V, generator=gen, device=device)
        off = -1.1 * torch.log(perm.double() + 1.0)
        h[..., d - 1] = 8.0
        W[d - 1, :] = (off / 8.0).float()
    h, W, Wg, A, Bt = (t.to(dt).contiguous() for t in (h, W, Wg, A, Bt))

    # --- target logits: noisy copy of a reference product (input synthesis only) ---
    P = L - 1
    u = _reference_product(h[:, 1:, :], W)  # [B, P, V] fp32
    kind = spec.agreement[0]
    if kind == "top1_linear":
        first, last = spec.agreement[1], spec.agreement[2]
        targets = [first + (last - first) * (p / max(1, P - 1)) for p in range(P)]
        sig = [_bisect_sigma(u[:, p, :], targets[p], "top1", gen, calib_reps) for p in range(P)]
        metric = "top1"
    else:
        s = _bisect_sigma(u.reshape(B * P, V), spec.agreement[1], kind, gen, calib_reps)
        sig = [s] * P
        metric = kind
    sig_t = torch.tensor(sig, dtype=torch.float32, device=device)  # sigma for positions 1..P
    noise = torch.randn(B, L, V, generator=gen, device=device)
    Z = torch.empty(B, L, V, dtype=torch.float32, device=device)
    Z[:, :P, :] = u + sig_t.view(1, P, 1) * noise[:, :P, :]
    Z[:, P, :] = u[:, P - 1, :] + sig_t[P - 1] * noise[:, P, :]
    Z = Z.to(dt).contiguous()

    with torch.no_grad():
        y = Z[:, :P, :].float().argmax(-1)
        if metric == "top1":
            hit = (y == u.argmax(-1))
        else:
            hit = (y.unsqueeze(-1) == u.topk(16, dim=-1).indices).any(-1)
        per_pos = hit.float().mean(0).tolist()
    del u
    meta = {"sigma": sig, "agreement_metric": metric, "agreement_target": list(spec.agreement),
            "agreement_realised_per_position": per_pos,
            "agreement_realised": float(sum(per_pos) / len(per_pos)), "device": str(device)}
    out = {"h": h, "W": W, "Wg": Wg, "A": A, "Bt": Bt, "x0": x0.to(torch.int32), "Z": Z,
           "meta": meta, "spec": spec}
    if spec.lmhead == "e4m3":
        out["Wq"], out["w_scale"] = quantize_lmhead_e4m3(W)
    return out


def quantize_lmhead_e4m3(W: torch.Tensor):
    """Input synthesis for the E4M3 LM head: W [d, V] -> (Wq [V, d] uint8 E4M3 bytes,
    w_scale [V] fp32), per vocabulary entry the smallest power-of-two scale 2^e with
    max|W[:, v]| <= 448 * 2^e (1 for an all-zero column), Wq = E4M3(W / scale) rounded to
    nearest even by torch's float8 cast."""
    Wt = W.float().t().contiguous()
    amax = Wt.abs().amax(dim=1)
    m, e = torch.frexp(amax)
    e = e - 9 + (m > 0.875).to(e.dtype)
    scale = torch.where(amax >= 2.0 ** -100, torch.ldexp(torch.ones_like(amax), e),
                        torch.ones_like(amax))
    Wq = (Wt / scale[:, None]).to(torch.float8_e4m3fn).view(torch.uint8).contiguous()
    return Wq, scale.float().contiguous()


def fresh_targets(data: dict, seed: int) -> torch.Tensor:
    """Another draw of target logits with the same noise scales (used to rotate Z buffers
    so successive timed steps do not reread one L2-resident copy)."""
    spec = data["spec"]
    gen = torch.Generator(device=data["Z"].device)
    gen.manual_seed(seed)
    noise = torch.randn(data["Z"].shape, generator=gen, device=data["Z"].device)
    scale = float(max(data["meta"]["sigma"]))
    return (data["Z"].float() + 0.25 * scale * noise).to(torch_dtype(spec)).contiguous()


@dataclasses.dataclass(frozen=True)
class ConvSpec:
    """Two-tap dynamic depthwise convolution inputs: x [B, L, d] (block row 0 the verified
    slot), one convolution's base kernels and correction map."""
    name: str
    B: int
    L: int
    d: int
    seed: int = 0

    def with_(self, **kw) -> "ConvSpec":
        return dataclasses.replace(self, **kw)


# the drafter width and block of the serving workload (B = 32 blocks of 8)
CONV_THROUGHPUT = ConvSpec("conv_B32_L8_d5120", B=32, L=8, d=5120, seed=11)
CONV_SMALL = ConvSpec("conv_B3_L5_d640", B=3, L=5, d=640, seed=12)


def conv_inputs(spec: ConvSpec, device="cpu") -> dict:
    """x ~ N(0, 1) in bf16; base kernels near a learned mix, base[0] ~ 1 + 0.1 N(0, 1) and
    base[1] ~ 0.5 + 0.1 N(0, 1) (fp32); the correction map Wc ~ N(0, 0.01 / d) in bf16, so
    each correction (one per 16 channels and tap) is about 0.1: small next to the base, as
    the pages describe it."""
    g = torch.Generator().manual_seed(spec.seed)
    d = spec.d
    x = torch.randn(spec.B, spec.L, d, generator=g).to(torch.bfloat16)
    base = torch.stack([1.0 + 0.1 * torch.randn(d, generator=g), 0.5 + 0.1 * torch.randn(d, generator=g)])
    Wc = (torch.randn(d // 8, d, generator=g) * (0.1 / math.sqrt(d))).to(torch.bfloat16)
    return {"x": x.to(device), "base": base.float().contiguous().to(device), "Wc": Wc.to(device)}


def to_numpy_bits(t: torch.Tensor):
    """Host numpy view of a tensor as the oracle takes it: bf16 -> uint16 bits, fp32 as is,
    integers as int32/int64."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view("uint16")
    return t.numpy()
