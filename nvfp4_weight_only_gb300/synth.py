"""Seeded synthetic inputs, shared by the tests, the benchmark and the smoke check.

This module only draws random numbers; it holds none of the NVFP4 arithmetic,
so feeding its tensors to both the CUDA path and the CPU oracle gives them
identical bytes without coupling the two.

Recipe (the decode workloads of the Atlas dense-FFN pages, with trained
checkpoints replaced by draws of the same shapes):
  * activations x ~ N(0, 1), rounded to bf16; optionally a seeded 1% of the
    positions multiplied by 20 (the outlier variant of the batch-M workload);
  * weights fp32 ~ N(0, 0.02), later quantised to NVFP4 by the library;
  * seeds: x uses seed 0 unless told otherwise; layer l uses 1000 + l with the
    gate / up / down projections as sub-streams 0 / 1 / 2;
  * block-scaled FP8 projections (stand-ins for an FP8 checkpoint, which the
    pages load as they are): E4M3 bytes of N(0, 1) * 448/4.5 draws (torch's
    float8_e4m3fn conversion, saturated at +-448) and an fp32 block grid of
    std * 4.5/448 * U(0.75, 1.25), one draw per 128 x 128 block, so the weights
    spread like N(0, std^2) and every block has its own scale.
"""
import torch

GATE, UP, DOWN = 0, 1, 2


def layer_seed(layer: int, proj: int) -> int:
    """Seed of projection `proj` (GATE/UP/DOWN) of layer `layer`."""
    return (1000 + int(layer)) * 4 + int(proj)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def weights_f32(N: int, K: int, seed: int, std: float = 0.02, device="cpu") -> torch.Tensor:
    """fp32 [N, K] ~ N(0, std^2)."""
    g = _gen(seed, device)
    return torch.randn((N, K), generator=g, dtype=torch.float32, device=device) * std


def fp8_weights(N: int, K: int, seed: int, std: float = 0.02, device="cpu"):
    """(E4M3 bytes uint8 [N, K], fp32 grid [ceil(N/128), ceil(K/128)]) as above."""
    g = _gen(seed, device)
    v = torch.randn((N, K), generator=g, dtype=torch.float32, device=device) * (448.0 / 4.5)
    codes = v.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
    shape = ((N + 127) // 128, (K + 127) // 128)
    u = torch.rand(shape, generator=g, dtype=torch.float32, device=device)
    return codes, (std * 4.5 / 448.0) * (0.75 + 0.5 * u)


def activations_bf16(M: int, K: int, seed: int = 0, outlier_frac: float = 0.0,
                     outlier_scale: float = 20.0, device="cpu") -> torch.Tensor:
    """bf16 [M, K] ~ N(0, 1), with `outlier_frac` of the positions scaled."""
    g = _gen(seed, device)
    x = torch.randn((M, K), generator=g, dtype=torch.float32, device=device)
    n_out = int(round(outlier_frac * M * K))
    if n_out > 0:
        idx = torch.randperm(M * K, generator=g, device=device)[:n_out]
        x.view(-1)[idx] *= outlier_scale
    return x.to(torch.bfloat16)


def bf16_bits(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (host copy)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")
