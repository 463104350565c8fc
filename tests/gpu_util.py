"""Helpers shared by the GPU parity tests (conversions and the attention
tolerance).  No method arithmetic lives here."""
import numpy as np
import torch

# Attention tolerance against the fp64 oracle for bf16 inputs (fp32
# accumulation, bf16 output): max |err| <= 1e-2 and relative L2 <= 5e-3.
ATOL_MAX = 1e-2
REL_L2 = 5e-3
# LSE is returned in fp32; |err| bound over a softmax of <= a few thousand terms.
LSE_ATOL = 2e-3


def bits(t):
    """bf16 tensor (any device) -> numpy uint16 bit patterns."""
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def u8(t):
    return t.detach().to("cpu").contiguous().view(torch.uint8).numpy()


def np_i32(t):
    return t.detach().to("cpu").numpy()


def cuda(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def check_attention(out_gpu, lse_gpu, out_ref, lse_ref, label=""):
    o = out_gpu.detach().float().cpu().numpy().astype(np.float64)
    err = np.abs(o - out_ref)
    max_abs = float(err.max()) if err.size else 0.0
    denom = float(np.sqrt((out_ref ** 2).sum()))
    rel = float(np.sqrt(((o - out_ref) ** 2).sum()) / denom) if denom > 0 else float(
        np.sqrt((o ** 2).sum()))
    assert max_abs <= ATOL_MAX, f"{label}: max abs err {max_abs}"
    assert rel <= REL_L2, f"{label}: rel L2 err {rel}"
    if lse_gpu is not None:
        l = lse_gpu.detach().cpu().numpy().astype(np.float64)
        fin = np.isfinite(lse_ref)
        assert (np.isfinite(l) == fin).all(), f"{label}: -inf pattern differs"
        assert (l[~fin] == -np.inf).all()
        if fin.any():
            lerr = float(np.abs(l[fin] - lse_ref[fin]).max())
            assert lerr <= LSE_ATOL, f"{label}: lse err {lerr}"
    return max_abs, rel
