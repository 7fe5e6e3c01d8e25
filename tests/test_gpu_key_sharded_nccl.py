"""dsa_indexer_key_sharded -- the binding's whole context-parallel path (this rank's shard
candidates, the all-gather, the merge) -- on a one-rank NCCL group: with a single rank the
shard is the whole key range, so the result must equal dsa_indexer_topk of the full scores,
bit for bit on integer-valued inputs.  Runs in a subprocess so the process group never
outlives the test.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CODE = r"""
import socket, numpy as np, torch, torch.distributed as dist
import sparse_attention_token_gb300 as dsa, workloads
s = socket.socket(); s.bind(("127.0.0.1", 0)); port = s.getsockname()[1]; s.close()
dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1,
                        device_id=torch.device("cuda", 0))
try:
    c = workloads.dense_case(300, 900, 64, 128, 128, q_pos0=600, integer=True, int_range=(-2, 2), seed=97)
    q, k, w = c.q.cuda(), c.k.cuda(), c.w.cuda()
    got = dsa.dsa_indexer_key_sharded(q, k, w, q_pos0=600, key_offset=0, topk_limit=128)
    sc = dsa.dsa_indexer_scores(q, k, w, q_pos0=600)
    ref = dsa.dsa_indexer_topk(sc, T=300, S=900, q_pos0=600, topk_limit=128)
    torch.cuda.synchronize()
    assert dsa.dsa_check_device_status() == dsa.DSA_OK
    assert np.array_equal(got.cpu().numpy(), ref.cpu().numpy())
    print("OK")
finally:
    dist.destroy_process_group()
"""


def test_key_sharded_one_rank_nccl_equals_unsharded():
    import __graft_entry__ as g
    g.build()
    r = subprocess.run([sys.executable, "-c", CODE], cwd=ROOT, capture_output=True, text=True, timeout=300,
                       env={**os.environ, "PYTHONPATH": ROOT, "NCCL_NVLS_ENABLE": "0"})
    assert r.returncode == 0 and "OK" in r.stdout, r.stdout[-2000:] + r.stderr[-2000:]
