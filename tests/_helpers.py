"""Shared helpers of the GPU parity tests: seeded inputs, host <-> device
conversions, and the oracle-side reference for each configuration."""
import numpy as np
import torch

import oracle
import synth


def dev():
    return torch.device("cuda", torch.cuda.current_device())


def bf16_to_dev(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev())


def bits_of(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def f32_of_bits(b: np.ndarray) -> np.ndarray:
    return oracle.bf16_bits_to_f32(b)


def activations_bf16(seed, M, K, p=0.0, factor=1.0, tensor=0):
    return synth.to_bf16_bits(synth.activations(seed, M, K, p, factor, tensor=tensor))


def quantised_weights(r9q, seed, N, K, tensor=0, check_oracle=True):
    """fp32 master weights -> (GPU) e4m3 + block scales.  With check_oracle the
    bytes and scales are compared with the oracle's (bit-exact)."""
    w = synth.weights(seed, N, K, tensor=tensor)
    wq, ws = r9q.r9q_quant_weight_block128(torch.from_numpy(w).to(dev()))
    torch.cuda.synchronize()
    if check_oracle:
        oq, os_ = oracle.quant_block128(w)
        assert np.array_equal(wq.cpu().numpy(), oq), "weight codes differ from the oracle"
        assert np.array_equal(ws.cpu().numpy(), os_), "weight scales differ from the oracle"
    return wq, ws


def assert_close(gpu_bf16_bits, ref_f32, what):
    ok, worst = oracle.tolerance_ok(f32_of_bits(gpu_bf16_bits), ref_f32)
    assert ok, f"{what}: outside |d| <= 8e-3|ref| + 1e-3 max|ref| (worst {worst:.3f} of the bound)"
    return worst
