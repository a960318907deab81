"""Test helpers: move seeded BF16 bits between numpy, the oracle and CUDA."""
import numpy as np
import torch

from oracle import formats as OF


def to_dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def to_f32(bits: np.ndarray) -> np.ndarray:
    return OF.bf16_bits_to_f32(bits)


def np_u8(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy().astype(np.uint8)


def np_f32(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy().astype(np.float32)


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of BF16 numbers at |x| (8 significant bits; 2^-133 at the bottom)."""
    _, e = np.frexp(np.abs(x))
    return np.ldexp(1.0, np.maximum(e - 8, -133))


def assert_gemm_close(got: np.ndarray, ref: np.ndarray, rel_fro: float = 1e-3, elem: float = 2e-2):
    """Relative Frobenius error <= rel_fro, and every |err| <= max(elem * rms(ref),
    one BF16 ulp of the reference element).

    The ulp term is the output format's own rounding step: the reference is the
    exact sum rounded once to BF16, the GPU rounds its FP32 accumulation to
    BF16, and near a rounding tie two correct results differ by one ulp, which
    for |ref| above ~2.5 rms exceeds 2e-2 * rms.
    """
    err = got - ref
    nref = np.linalg.norm(ref)
    rms = nref / np.sqrt(ref.size) if ref.size else 0.0
    rel = np.linalg.norm(err) / max(nref, 1e-300)
    assert rel <= rel_fro, f"relative Frobenius error {rel:.3e} > {rel_fro}"
    bound = np.maximum(elem * rms, bf16_ulp(ref))
    bad = np.abs(err) > bound
    assert not bad.any(), (f"{int(bad.sum())} elements beyond max(2e-2*rms, 1 bf16 ulp); worst |err| "
                           f"{np.abs(err).max():.3e}, rms {rms:.3e}")
    return rel, (np.abs(err).max() / max(rms, 1e-300)) if err.size else 0.0
