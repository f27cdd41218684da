"""The allocation-free expert MLP entry point (for callers that cannot
allocate device memory where they run the MLP) against the regular entry
point, through the C ABI.  It keeps h in a scratch array inside the library, so
two calls in a row with different inputs also check that nothing of the first
call leaks into the second.  Collected last on purpose (file name)."""
import numpy as np
import pytest
import torch

import oracle
from _helpers import activations_bf16, bf16_to_dev, bits_of, dev, f32_of_bits, quantised_weights

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def r9q():
    import __graft_entry__
    __graft_entry__.build()
    import block_scaled_fp8_x128_gb300 as lib
    return lib


@pytest.mark.parametrize("weight_only", [False, True])
def test_noalloc_matches_regular_entry_point_two_calls(r9q, weight_only):
    M, H, I, Ho = 8, 4096, 1536, 4096          # the decode expert MLP shape
    wgu, sgu = quantised_weights(r9q, 3, 2 * I, H, tensor=1, check_oracle=False)
    wdn, sdn = quantised_weights(r9q, 3, Ho, I, tensor=2, check_oracle=False)
    flags = r9q.R9Q_MLP_WEIGHT_ONLY if weight_only else 0
    for call, seed in enumerate((31, 32)):     # two calls in a row, different inputs
        x = bf16_to_dev(activations_bf16(seed, M, H))
        hq = None if weight_only else torch.empty((M, I), dtype=torch.uint8, device=dev())
        hs = None if weight_only else torch.empty((M, I // 128), dtype=torch.float32, device=dev())
        y_na = r9q.r9q_gate_up_swiglu_down_noalloc(x, wgu, sgu, wdn, sdn, hq=hq, hs=hs, flags=flags)
        y_ref = r9q.r9q_gate_up_swiglu_down(x, wgu, sgu, wdn, sdn, flags=flags)
        torch.cuda.synchronize()
        ok, worst = oracle.tolerance_ok(f32_of_bits(bits_of(y_na)), f32_of_bits(bits_of(y_ref)))
        assert ok, f"call {call}: outside the output tolerance (worst {worst:.3f} of the bound)"
        assert torch.equal(y_na.view(torch.int16), y_ref.view(torch.int16)), f"call {call}: not bit-identical"
    assert r9q.r9q_last_device_error() == 0


@pytest.mark.parametrize("weight_only", [False, True])
def test_noalloc_back_to_back_with_programmatic_launch(r9q, weight_only):
    """Programmatic dependent launch on: the next call's gate_up kernel may
    start while the previous call's down GEMM still reads h from the shared
    scratch, and must not write h before that GEMM has finished.  Four calls
    with different inputs are queued on one stream without a synchronise in
    between; each output must equal the regular entry point's, bit for bit."""
    M, H, I, Ho = 8, 4096, 1536, 4096
    wgu, sgu = quantised_weights(r9q, 3, 2 * I, H, tensor=1, check_oracle=False)
    wdn, sdn = quantised_weights(r9q, 3, Ho, I, tensor=2, check_oracle=False)
    flags = r9q.R9Q_MLP_WEIGHT_ONLY if weight_only else 0
    xs = [bf16_to_dev(activations_bf16(40 + i, M, H, 0.01, 20.0)) for i in range(4)]
    refs = [r9q.r9q_gate_up_swiglu_down(x, wgu, sgu, wdn, sdn, flags=flags) for x in xs]
    torch.cuda.synchronize()
    prev = r9q.r9q_set_pdl(True)
    try:
        outs = [r9q.r9q_gate_up_swiglu_down_noalloc(x, wgu, sgu, wdn, sdn, flags=flags) for x in xs]
        torch.cuda.synchronize()
    finally:
        r9q.r9q_set_pdl(prev)
    for i, (y, ref) in enumerate(zip(outs, refs)):
        assert torch.equal(y.view(torch.int16), ref.view(torch.int16)), f"call {i}: not bit-identical"
    assert r9q.r9q_last_device_error() == 0


def test_noalloc_rejects_oversized_and_unfused(r9q):
    M, H, I, Ho = 512, 256, 2048, 256           # M * I = 1,048,576 > 524,288
    x = torch.zeros((M, H), dtype=torch.bfloat16, device=dev())
    wgu = torch.zeros((2 * I, H), dtype=torch.uint8, device=dev())
    sgu = torch.zeros((2 * I // 128, H // 128), dtype=torch.float32, device=dev())
    wdn = torch.zeros((Ho, I), dtype=torch.uint8, device=dev())
    sdn = torch.zeros((Ho // 128, I // 128), dtype=torch.float32, device=dev())
    with pytest.raises(r9q.R9QError) as e:
        r9q.r9q_gate_up_swiglu_down_noalloc(x, wgu, sgu, wdn, sdn)
    assert e.value.code == -4
    with pytest.raises(r9q.R9QError) as e:
        r9q.r9q_gate_up_swiglu_down_noalloc(x[:8], wgu, sgu, wdn, sdn, flags=r9q.R9Q_MLP_UNFUSED)
    assert e.value.code == -8
