"""GPU checks shaped like the kernel-level checks printed on the pages
("[ROCm][Spec Decode] Add Aiter MLA decode support non-causal draft block",
section on the kernel checks):

* an fp8 cache with 16 heads, draft blocks of 4 and 8 tokens: the non-causal call
  matches the non-causal reference and stays far from the causal one, so the mask
  that runs is the one asked for;
* a bf16 cache over 8, 12, 16, 24 and 32 heads and blocks of 1 to 16 tokens
  (causal), every combination within the parity tolerance.

The pages' deviation figures come from their own data, which they do not describe,
so the checks here assert the same properties (reference agreement, mask
separation) rather than those numbers.
"""
import dataclasses

import numpy as np
import pytest

import mla_inputs as mi
from oracle import mla_oracle as mo

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a GPU", allow_module_level=True)

import token_mla_paged_gb300 as m  # noqa: E402
from tests import harness as hz  # noqa: E402


@pytest.mark.parametrize("block", [4, 8])
def test_fp8_non_causal_runs_the_mask_asked_for(block):
    w = mi.make_workload(f"nc_fp8_T{block}", batch=4, num_heads=16, q_lens=[block] * 4,
                         kv_lens=[40, 64, 129, 700], kv_dtype="fp8", causal=False, seed=300 + block)
    O, L, runner = hz.run(w, algo=m.MLA_ALGO_TENSOR)
    assert hz.device_error(runner) == (0, 0)
    O_nc, L_nc = mo.mla_decode_workload(w)
    hz.assert_close(O, L, O_nc, L_nc, "fp8")
    O_c, _ = mo.mla_decode_workload(dataclasses.replace(w, causal=True))
    d_nc = np.abs(O - O_nc).max()
    d_c = np.abs(O - O_c).max()
    assert d_c > 2e-2 and d_c > 3 * d_nc, (d_nc, d_c)


@pytest.mark.parametrize("heads", [8, 12, 16, 24, 32])
def test_bf16_heads_and_blocks_grid(heads):
    for block in range(1, 17):
        w = mi.make_workload(f"grid_H{heads}_T{block}", batch=2, num_heads=heads, q_lens=[block, block],
                             kv_lens=[257, 40 + block], kv_dtype="bf16", causal=True,
                             seed=1000 + heads * 17 + block)
        O, L, runner = hz.run(w, algo=m.MLA_ALGO_TENSOR)
        assert hz.device_error(runner) == (0, 0)
        Oref, Lref = mo.mla_decode_workload(w)
        hz.assert_close(O, L, Oref, Lref, "bf16", what=f"H={heads} T={block}")
