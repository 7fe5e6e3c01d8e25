"""The front-end's fused q projection: with 512 tokens or more the q projection finishes
its rows (RoPE, and on the FP8 path the rotation and quantisation) in the epilogue of
the tensor-core product instead of writing fp32 rows for the q row kernel.  Checked
against the fp64 oracle with the same tolerances as the other front-end tests, for both
RoPE layouts, both caches, rope_dim 0 / 64 / 128, a token count that leaves a partial
128-token tile, and a head count whose weight projection is narrower than one tile.
"""
import numpy as np
import pytest

import workloads

pytestmark = pytest.mark.gpu

dsa = pytest.importorskip("sparse_attention_token_gb300")

from tests.test_gpu_frontend import (assert_bf16_close, assert_e4m3_close, assert_w_close, cache_rows,  # noqa: E402
                                     run_gpu, run_oracle)


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


@pytest.mark.parametrize("fp8,interleaved,rope_dim,H", [(True, False, 64, 64), (True, True, 128, 16),
                                                        (False, False, 128, 32), (False, True, 64, 8),
                                                        (True, False, 0, 4)])
def test_fused_q_projection(fp8, interleaved, rope_dim, H):
    c = workloads.frontend_case(700, 256, 320, H, rope_dim=rope_dim, fp8=fp8, bias=True, pos0=300, seed=31 + H)
    got, ref = run_gpu(c, interleaved), run_oracle(c, interleaved)
    assert got["status"] == dsa.DSA_OK
    if fp8:
        qc = assert_e4m3_close(got["q"], got["q_scale"], ref["q"], ref["q_scale"].astype(np.float64), "q")
        assert (qc == ref["q_codes"]).mean() > 0.99
    else:
        assert_bf16_close(got["q"], ref["q"], "q")
    assert_w_close(got["w"], c, ref["w"])
    rows, sc, valid = cache_rows(got, c)
    if fp8:
        kc = assert_e4m3_close(rows, sc, ref["k"][valid], ref["k_scale"][valid].astype(np.float64), "k")
        assert (kc == ref["k_codes"][valid]).mean() > 0.99
    else:
        assert_bf16_close(rows, ref["k"][valid], "k")
