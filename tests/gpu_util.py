"""Helpers for the GPU parity tests: host copies and the stated tolerances."""
import numpy as np
import torch

# Tolerances (stated for the method: logits relative to the row's max |logit|;
# indices bit-exact; attention output max-abs and LSE abs), plus a relative RMS
# bound on the output that catches real bugs the loose max-abs would not.
LOGIT_REL = 1e-3
O_MAX_ABS = 2e-2
LSE_ABS = 1e-3
O_REL_RMS = 1e-2


def bits16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def lib():
    import sparse_attention_02_gb300 as dsa

    dsa.load_library()
    return dsa


def check_logits(got: np.ndarray, ref: np.ndarray, pos: np.ndarray):
    """Compare indexer rows over s <= pos[r]."""
    worst = 0.0
    for r in range(ref.shape[0]):
        n = int(pos[r]) + 1
        if n <= 0:
            continue
        m = np.abs(ref[r, :n]).max()
        err = np.abs(got[r, :n] - ref[r, :n]).max()
        assert np.all(np.isfinite(got[r, :n])), f"row {r}: non-finite logits"
        assert err <= LOGIT_REL * m + 1e-30, f"row {r}: err {err} vs max {m}"
        worst = max(worst, err / max(m, 1e-30))
    return worst


def check_attention(o: np.ndarray, l: np.ndarray, o_ref: np.ndarray, l_ref: np.ndarray):
    assert np.all(np.isfinite(o)), "non-finite attention output"
    fin = np.isfinite(l_ref)
    assert np.array_equal(fin, np.isfinite(l)), "LSE finiteness differs"
    err_o = np.abs(o - o_ref).max() if o.size else 0.0
    err_l = np.abs(l[fin] - l_ref[fin]).max() if fin.any() else 0.0
    rms = np.sqrt(np.mean((o - o_ref) ** 2)) / max(np.sqrt(np.mean(o_ref ** 2)), 1e-30)
    assert err_o <= O_MAX_ABS, f"O max-abs err {err_o}"
    assert err_l <= LSE_ABS, f"LSE abs err {err_l}"
    assert rms <= O_REL_RMS, f"O relative RMS err {rms}"
    return err_o, err_l, rms
