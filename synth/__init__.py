"""Seeded synthetic inputs for the routed-expert MoE FFN workloads.

Draws only: this module holds none of the quantization, routing or GEMM
arithmetic. Both the CUDA path and the CPU oracle consume what it returns (the
oracle as host copies). Every tensor comes from a torch.Generator seeded from
(workload seed, tag), so a (seed, tag, device) triple always yields the same
values; CPU and CUDA generators give different streams, so a test draws once on
one device and hands copies to both sides.

Distributions follow the workloads of the pages:
* activations bf16 N(0, 1);
* expert weights float32 N(0, 0.02) (quantized afterwards by whoever consumes them);
* routes: per token, top-k distinct experts drawn uniformly without replacement;
  a chosen number of a token's slots set to -1 (inactive, e.g. CPU-assigned);
* routing weights: softmax of N(0, 1) logits over the k slots (the router's output;
  not renormalised when slots are inactive);
* gather workload: random FP8 bytes, fp32 scales U(1e-3, 1), randint maps.
"""
import torch

_MASK64 = (1 << 64) - 1


def splitmix64(x: int) -> int:
    """SplitMix64 output function (Steele, Lea, Flood 2014), used to derive sub-seeds."""
    x = (x + 0x9E3779B97F4A7C15) & _MASK64
    z = x
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
    return z ^ (z >> 31)


def sub_seed(seed: int, *tags) -> int:
    s = seed & _MASK64
    for t in tags:
        if isinstance(t, str):
            t = sum(ord(c) << (8 * (i % 7)) for i, c in enumerate(t))
        s = splitmix64(s ^ (int(t) & _MASK64))
    return s & ((1 << 63) - 1)


def _gen(seed, device, *tags):
    g = torch.Generator(device=device)
    g.manual_seed(sub_seed(seed, *tags))
    return g


def activations_bf16(tokens, hidden, seed, device="cpu"):
    """x ~ N(0, 1), rounded to bf16: [tokens, hidden]."""
    g = _gen(seed, device, "x")
    return torch.randn(tokens, hidden, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def expert_weight_fp32(n, k, seed, expert, tag, device="cpu", std=0.02):
    """One expert's raw weight matrix [n, k] ~ N(0, std), float32. tag names the matrix."""
    g = _gen(seed, device, "w", tag, expert)
    return torch.randn(n, k, generator=g, device=device, dtype=torch.float32) * std


def routes(tokens, topk, num_experts, seed, active_per_token=None, device="cpu"):
    """expert_ids [tokens, topk] int32: distinct experts per token, uniform without replacement.

    active_per_token: None (all active), an int, or a list per token; the inactive
    slots (chosen by seed) hold -1.
    """
    g = _gen(seed, "cpu", "routes")
    ids = torch.empty(tokens, topk, dtype=torch.int32)
    for t in range(tokens):
        ids[t] = torch.randperm(num_experts, generator=g)[:topk].to(torch.int32)
    if active_per_token is not None:
        for t in range(tokens):
            a = active_per_token if isinstance(active_per_token, int) else active_per_token[t]
            off = torch.randperm(topk, generator=g)[: topk - a]
            ids[t, off] = -1
    return ids.to(device)


def routes_fast(tokens, topk, num_experts, seed, device="cpu"):
    """Like routes() with every slot active, vectorised (for thousands of tokens)."""
    g = _gen(seed, "cpu", "routes-fast")
    keys = torch.rand(tokens, num_experts, generator=g)
    ids = torch.argsort(keys, dim=1)[:, :topk].to(torch.int32)
    return ids.to(device)


def routing_weights(tokens, topk, seed, device="cpu"):
    """softmax over the k slots of N(0, 1) logits, float32 [tokens, topk]."""
    g = _gen(seed, "cpu", "logits")
    logits = torch.randn(tokens, topk, generator=g, dtype=torch.float64)
    return torch.softmax(logits, dim=1).to(torch.float32).to(device)


def random_bytes(rows, cols, seed, tag="bytes", device="cpu"):
    g = _gen(seed, "cpu", tag)
    return torch.randint(0, 256, (rows, cols), generator=g, dtype=torch.uint8).to(device)


def uniform_f32(rows, cols, lo, hi, seed, tag="uniform", device="cpu"):
    g = _gen(seed, "cpu", tag)
    return (torch.rand(rows, cols, generator=g, dtype=torch.float64) * (hi - lo) + lo).to(torch.float32).to(device)


def randint_map(n, high, seed, tag="map", device="cpu"):
    g = _gen(seed, "cpu", tag)
    if n == 0:
        return torch.zeros(0, dtype=torch.int32, device=device)
    return torch.randint(0, high, (n,), generator=g, dtype=torch.int64).to(torch.int32).to(device)


def subsample(n, count, seed):
    """`count` distinct indices of range(n), sorted, drawn by seed."""
    g = _gen(seed, "cpu", "subsample")
    return torch.sort(torch.randperm(n, generator=g)[:count]).values.tolist()
