"""Shared helpers for the GPU parity tests (no method arithmetic here)."""
import numpy as np
import torch

TOL_ABS, TOL_REL = 0.02, 0.01  # |C - C_ref| <= 0.02 + 0.01 |C_ref|


def bits16(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (CPU copy)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def assert_within_tol(got_bf16: torch.Tensor, ref_bits: np.ndarray, what: str = ""):
    import oracle
    ref = oracle.bf16_to_f32(ref_bits).astype(np.float64)
    got = got_bf16.float().cpu().numpy().astype(np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    err = np.abs(got - ref)
    bad = err > TOL_ABS + TOL_REL * np.abs(ref)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; first {idx.tolist()} "
                             f"got {got[tuple(idx[0])]} ref {ref[tuple(idx[0])]}")


def requires_gpu():
    import pytest
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def trace_buffer(words_per_cta: int) -> torch.Tensor:
    """Zeroed device buffer for the per-CTA trace: one record per SM of the current device
    (the kernels launch at most one CTA per SM)."""
    nsm = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    return torch.zeros(nsm * words_per_cta, dtype=torch.int64, device="cuda")
