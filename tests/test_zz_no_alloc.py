"""The allocation-free selector entry point (needs a GB300).

bsa_topk_select_noalloc serves callers that cannot call cudaMalloc: code
running under a CUDA-graph capture mode that forbids allocation, plugins
whose host engine owns all device memory, loops that must not enter the
allocator.  It keeps the split path's scratch in the library's own device
array instead of a caller workspace.  These tests call it through the C ABI
and check it against the regular entry point and against the CPU oracle,
twice in a row (the array keeps the previous call's contents), on workloads
that need scratch and on one that does not.  The file is named so that
pytest collects it last.
"""
import numpy as np
import pytest
import torch

import block_sparse_attention_topk_gb300 as bsa
import oracle
import synth

pytestmark = pytest.mark.gpu


def _split_case(T, H, M, K, dtype, seed):
    scores = synth.normal_scores((T, H, M), dtype, seed=seed)
    synth.inject_specials(scores, seed=seed + 1)
    nvp = torch.from_numpy(np.linspace(1, M + 7, T).astype(np.int32))
    return scores, nvp


@pytest.mark.parametrize("T,H,M,K,dtype", [
    (24, 2, 8192, 16, torch.bfloat16),   # split rows: scratch in use
    (16, 1, 4096, 64, torch.float32),    # split rows, another layout of the scratch
    (40, 3, 300, 16, torch.bfloat16),    # no scratch needed
])
def test_noalloc_matches_regular_entry_point(cuda_device, T, H, M, K, dtype):
    scores, nvp = _split_case(T, H, M, K, dtype, seed=M + K)
    s = scores.to(cuda_device)
    n = nvp.to(cuda_device)
    dt = bsa.BSA_DTYPE_BF16 if dtype == torch.bfloat16 else bsa.BSA_DTYPE_FP32
    need = bsa.bsa_topk_workspace_bytes(T, H, M, K, dt)
    if M >= 4096:
        assert need > 0, "this case should exercise the scratch"
    ref = bsa.bsa_topk_select(s, n, K, 1, 2)
    torch.cuda.synchronize()
    want = oracle.topk_select(scores, nvp.numpy(), K, 1, 2)
    for _ in range(2):
        got = bsa.bsa_topk_select_noalloc(s, n, K, 1, 2)
        torch.cuda.synchronize()
        assert torch.equal(got, ref)
        assert np.array_equal(got.cpu().numpy(), want)


def test_noalloc_rejects_requests_beyond_its_scratch(cuda_device):
    T, H, M, K = 64, 1, 65536, 1024
    dt = bsa.BSA_DTYPE_BF16
    need = bsa.bsa_topk_workspace_bytes(T, H, M, K, dt)
    assert need > bsa.NOALLOC_SCRATCH_BYTES
    s = torch.zeros((T, H, M), dtype=torch.bfloat16, device=cuda_device)
    n = torch.full((T,), M, dtype=torch.int32, device=cuda_device)
    with pytest.raises(bsa.BsaError) as e:
        bsa.bsa_topk_select_noalloc(s, n, K, 1, 1)
    assert e.value.status == -8
