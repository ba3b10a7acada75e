"""The library's host expert FFN (what its cold-route workers run) against the oracle, on the CPU.

Both compute y = Wd (SiLU(Wg x) * (Wu x)) in fp32 from the same MXFP4 record; they differ only in the order of
the fp32 sums (the library sums each 32-column block in eight interleaved partial sums), so they agree to a few
fp32 roundings of the row sums."""
import numpy as np
import pytest

import oracle
from expert_offload_moe_gb300 import moe, synth


def _check(H, I, n_experts, n_inputs, seed=0):
    recs = synth.expert_records(seed, 0, n_experts, H, I)
    for e in range(n_experts):
        for s in range(n_inputs):
            x = synth.activations(seed, 0, 40 + s, 1, H)[0]
            got = moe.host_expert_ffn(recs[e], H, I, x)
            ref = oracle.expert_ffn(recs[e], H, I, x)
            # a sum that cancels to near zero moves by roundings the size of its terms, not of itself: the
            # floor is 10% of the row's RMS (observed differences stay below 2e-6 of the RMS)
            floor = 1e-1 * np.sqrt(np.mean(ref.astype(np.float64) ** 2))
            err = np.abs(got.astype(np.float64) - ref) / np.maximum(np.abs(ref), floor)
            assert err.max() <= 1e-4, (H, I, e, s, float(err.max()))


def test_host_ffn_tiny():
    _check(256, 128, 4, 3)


def test_host_ffn_e512_shape():
    _check(2048, 512, 2, 2)


def test_host_ffn_gptoss_shape():
    _check(2880, 2880, 1, 1)


def test_host_ffn_rejects_bad_shapes():
    rec = np.zeros(synth.expert_bytes(256, 128), dtype=np.uint8)
    with pytest.raises(moe.MoeError):
        moe.host_expert_ffn(rec, 250, 128, np.zeros(250, dtype=np.uint16))
