"""GPU parity of the E4M3 state quantize-dequantize (delta_rule_state_fp8_qdq) with the oracle:
bit-exact, since the codes are decided in float32 on both sides.  States with partial value
tiles, all-zero tiles, a wide dynamic range (subnormal codes), in place and out of place."""
import numpy as np
import pytest
import torch

from oracle import fp8_qdq as Q
from linear_recurrent_rnn_gb300 import librglru as R

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape,block_v", [((3, 2, 128, 100), 64), ((5, 64, 64), 64),
                                           ((2, 32, 37), 8), ((1, 1, 1), 1)])
def test_state_qdq_is_bit_exact(shape, block_v):
    rng = np.random.default_rng(sum(shape) + block_v)
    st = (rng.standard_normal(shape) * np.exp(rng.uniform(-8, 4, shape))).astype(np.float32)
    if shape[-1] > block_v:
        st[..., :block_v] = 0.0 if len(shape) == 3 else st[..., :block_v]
    if len(shape) == 4:
        st[1, 0, :, block_v:] = 0.0              # an all-zero (partial) tile
    ref = Q.state_fp8_qdq(st, block_v)
    d = torch.from_numpy(st).cuda()
    out = torch.empty_like(d)
    R.delta_rule_state_fp8_qdq(d, out, block_v)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out.cpu().numpy(), ref)
    R.delta_rule_state_fp8_qdq(d, d, block_v)         # in place
    torch.cuda.synchronize()
    np.testing.assert_array_equal(d.cpu().numpy(), ref)
