"""Shared helpers of the GPU parity tests (the CPU oracle against libnc)."""
import numpy as np
import torch

REL_L2_GATE = 5e-4  # the parity gate for floating-point outputs


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def f32(t):
    return t.detach().float().cpu().numpy()


def weights_both(shape, seed=0):
    """The seeded weights generated on the GPU (fast), plus a CPU copy for the
    oracle. The generator's integer arithmetic gives the same bits on either
    device (test_gpu_model checks this)."""
    from transformer_decode_gb300 import synth
    wd = synth.model_weights(shape, seed=seed, device="cuda")
    return wd, to_device(wd, "cpu")


def to_device(weights, device="cuda"):
    """The generator's weight dict with every tensor moved to the device."""
    out = {k: (None if v is None else v.to(device)) for k, v in weights.items() if k != "layers"}
    out["layers"] = [{k: (None if v is None else v.to(device)) for k, v in lw.items()}
                     for lw in weights["layers"]]
    return out


def bf16_bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def token_agrees(gpu_tok, oracle_logits, observed_rel_l2):
    """Greedy agreement with the near-tie rule: a different token is accepted
    only when the oracle's own top-2 gap is below 4 * (observed logit rel-L2)
    * max|logit|, i.e. both answers are within the measured error."""
    o = np.asarray(oracle_logits, np.float64)
    best = int(np.argmax(o))
    if gpu_tok == best:
        return True
    gap = o[best] - o[gpu_tok]
    return gap <= 4 * observed_rel_l2 * np.abs(o).max()


def guarded(n, dtype=torch.float32, guard=64, device="cuda"):
    """A NaN-filled buffer of n elements with guard words on both sides.
    Returns (view, check) where check() asserts the guards are intact."""
    buf = torch.full((n + 2 * guard,), float("nan"), dtype=dtype, device=device) \
        if dtype.is_floating_point else torch.full((n + 2 * guard,), -99, dtype=dtype, device=device)
    sentinel = 12345.0 if dtype.is_floating_point else 77
    buf[:guard] = sentinel
    buf[guard + n:] = sentinel
    view = buf[guard:guard + n]

    def check():
        assert bool((buf[:guard] == sentinel).all()), "write before the output"
        assert bool((buf[guard + n:] == sentinel).all()), "write past the output"
    return view, check
