"""dsa_indexer_static: the fused indexer for callers that cannot allocate device memory.

Plugin hosts that only pass tensors and serving loops that forbid allocation during
a step cannot give the library a workspace; this entry point keeps its scratch in a
fixed library-owned device array instead.  The tests call it through the C ABI on
several problems in a row -- bf16, e4m3, and bf16 queries against an e4m3 cache (the
path that also keeps the split query rows in the scratch) -- and check each result
against dsa_indexer with a caller workspace (integer-valued inputs: the results must
be identical), check that a repeated call changes neither torch's allocations nor the
device's free memory, and check that a problem needing more scratch than the
built-in maximum is refused.
This file is collected last so a failure here never hides another test's result.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

dsa = pytest.importorskip("sparse_attention_token_gb300")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


def _on_device(pc):
    to = lambda t: None if t is None else t.to("cuda")
    return dict(q=to(pc.q), w=to(pc.w), k_cache=to(pc.k_cache), cu_q_lens=to(pc.cu_q_lens),
                seq_lens=to(pc.seq_lens), block_tables=to(pc.block_tables), q_scale=to(pc.q_scale),
                k_scale_cache=to(pc.k_scale_cache))


def _static_call(d, pc, memory=None):
    """Call dsa_indexer_static through the C ABI; the args carry no workspace.  With
    ``memory`` (a list), append torch's allocated bytes and the device's free bytes
    taken just before and just after the call itself."""
    a, keep = dsa.make_indexer_args(d["q"], d["w"], d["k_cache"], d["cu_q_lens"], d["seq_lens"],
                                    d["block_tables"], max_seq_len=pc.max_seq_len, topk_limit=pc.topk_limit,
                                    q_scale=d["q_scale"], k_scale_cache=d["k_scale_cache"],
                                    workspace=torch.empty(0, dtype=torch.uint8, device="cuda"))
    a.workspace, a.workspace_bytes = None, 0
    fn = dsa.lib().dsa_indexer_static
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(dsa.dsa_indexer_args), ctypes.c_void_p]
    stream = torch.cuda.current_stream()
    if memory is not None:
        torch.cuda.synchronize()
        memory.append((torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0]))
    st = fn(ctypes.byref(a), stream.cuda_stream)
    if memory is not None:
        torch.cuda.synchronize()
        memory.append((torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0]))
    return st, keep[8]


def _workspace_call(d, pc):
    return dsa.dsa_indexer(d["q"], d["w"], d["k_cache"], d["cu_q_lens"], d["seq_lens"], d["block_tables"],
                           max_seq_len=pc.max_seq_len, topk_limit=pc.topk_limit, q_scale=d["q_scale"],
                           k_scale_cache=d["k_scale_cache"])


def test_static_workspace_matches_caller_workspace_twice():
    first = workloads.paged_case([3000, 700, 64, 1], [1, 1, 1, 1], 64, 128, 512, page_size=64,
                                 integer=True, seed=41)
    second = workloads.paged_case([1500, 900], [300, 5], 64, 128, 256, page_size=64, q_dtype="fp8_e4m3",
                                  k_dtype="fp8_e4m3", integer=True, seed=42)
    # decode rows with bf16 queries against an e4m3 cache: the split query rows live in the scratch too
    third = workloads.paged_case([2500, 4100, 333, 64, 1], [1] * 5, 64, 128, 512, page_size=64,
                                 q_dtype="bf16", k_dtype="fp8_e4m3", integer=True, seed=44)
    for pc in (first, second, third):
        d = _on_device(pc)
        st, got = _static_call(d, pc)
        assert st == dsa.DSA_OK, dsa.dsa_status_string(st)
        ref = _workspace_call(d, pc)
        torch.cuda.synchronize()
        assert dsa.dsa_check_device_status() == dsa.DSA_OK
        assert np.array_equal(got.cpu().numpy(), ref.cpu().numpy())


def test_static_call_allocates_nothing():
    pc = workloads.paged_case([2500, 4100, 333, 64, 1], [1] * 5, 64, 128, 512, page_size=64,
                              q_dtype="bf16", k_dtype="fp8_e4m3", integer=True, seed=45)
    d = _on_device(pc)
    st, first = _static_call(d, pc)              # warm-up: loads the kernels it needs
    assert st == dsa.DSA_OK, dsa.dsa_status_string(st)
    memory = []
    st, again = _static_call(d, pc, memory)
    assert st == dsa.DSA_OK, dsa.dsa_status_string(st)
    (alloc0, free0), (alloc1, free1) = memory
    assert alloc1 == alloc0, "torch allocated during the call"
    assert free1 == free0, "device free memory changed during the call"
    assert np.array_equal(first.cpu().numpy(), again.cpu().numpy())


def test_static_workspace_refuses_oversized_problems():
    # the score rows are max_seq_len long: 64 decode rows with max_seq_len 200000 (one context
    # of 200000 keys sets it) need 64 * 200000 * 4 B of scores, more than the 24 MiB built in
    pc = workloads.paged_case([200000] + [1] * 63, [1] * 64, 64, 128, 64, page_size=64, integer=True,
                              seed=43)
    d = _on_device(pc)
    st, _ = _static_call(d, pc)
    assert st == dsa.DSA_ERR_WORKSPACE
