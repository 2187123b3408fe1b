"""mkv_compress_noalloc: the compression path for callers that cannot
allocate device memory (a plugin that only receives input/output pointers and
a stream, a server whose memory planner forbids allocations while serving, a
latency-critical path that cannot take cudaMalloc's implicit device
synchronisation). It uses the library's own fixed 32 MiB scratch array
instead of a caller workspace.

The test calls it through the C ABI twice in a row, on different problems,
and checks each result against mkv_compress on the same inputs. Both calls
run the same kernels, so kept counts, indices and compacted rows must match
bit for bit. The second call checks that the contents the first call left
in the shared array do not leak into the next result. This file is named
to be collected last, so a run that stops at its first failure has already
run every other test.
"""
import pytest
import torch

import geometric_kv_cache_gb300 as mkv
import synthkv


def _reference(K, V, ratio, mode, window, lens, ks):
    Ko = torch.zeros((K.shape[0], K.shape[1], ks, 128), dtype=torch.bfloat16, device="cuda")
    Vo = torch.zeros_like(Ko)
    idx = torch.full((K.shape[0], K.shape[1], ks), -1, dtype=torch.int32, device="cuda")
    kept = torch.full((K.shape[0], K.shape[1]), -1, dtype=torch.int32, device="cuda")
    ws = mkv.workspace_for(K, window, lens)
    mkv.mkv_compress(K, V, ratio, mode, window, ks, Ko, Vo, idx, kept, ws, lens)
    assert mkv.mkv_device_status(ws) == 0
    return Ko, Vo, idx, kept


def _no_alloc(K, V, ratio, mode, window, lens, ks):
    Ko = torch.zeros((K.shape[0], K.shape[1], ks, 128), dtype=torch.bfloat16, device="cuda")
    Vo = torch.zeros_like(Ko)
    idx = torch.full((K.shape[0], K.shape[1], ks), -1, dtype=torch.int32, device="cuda")
    kept = torch.full((K.shape[0], K.shape[1]), -1, dtype=torch.int32, device="cuda")
    status = torch.full((1,), 0x7F, dtype=torch.int32, device="cuda")
    mkv.mkv_compress_noalloc(K, V, ratio, mode, window, ks, Ko, Vo, idx, kept, status, lens)
    torch.cuda.synchronize()
    return Ko, Vo, idx, kept, int(status.item())


@pytest.mark.gpu
def test_no_alloc_matches_mkv_compress_on_two_calls_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cases = [
        # ragged lengths, cosine score, per-window centroids
        (synthkv.WORKLOADS["ragged-b8-llama-kv-t8k-32k"].scaled("noalloc-a", layers=2, batch=3, heads=4,
                                                                 t_max=20000, t_min=3000), "cosine", 4096, 0.3),
        # uniform lengths, L2 score, global centroid, another ratio
        (synthkv.WORKLOADS["llama3.1-8b-kv-t16k"].scaled("noalloc-b", layers=4), "l2", 0, 0.5),
    ]
    for w, mode, window, ratio in cases:
        K, V, lens = synthkv.make_kv(w, seed=7, device="cuda")
        ks = mkv.mkv_num_keep(w.t_max, ratio)
        ref = _reference(K, V, ratio, mode, window, lens, ks)
        got = _no_alloc(K, V, ratio, mode, window, lens, ks)
        assert got[4] == 0, f"device status {got[4]:#x}"
        Ko, Vo, idx, kept = ref
        assert torch.equal(got[3], kept)
        live = torch.arange(ks, device="cuda")[None, None, :] < kept[..., None]
        assert torch.equal(torch.where(live, got[2], -1), torch.where(live, idx, -1))
        assert torch.equal(torch.where(live[..., None], got[0], 0), torch.where(live[..., None], Ko, 0))
        assert torch.equal(torch.where(live[..., None], got[1], 0), torch.where(live[..., None], Vo, 0))


def test_no_alloc_refuses_problems_beyond_its_scratch():
    # 512 heads x 32K tokens need more scratch than the fixed 32 MiB array:
    # the call returns MKV_ERR_UNSUPPORTED on the host, before touching any
    # pointer (so none is needed here, and no GPU).
    shape = mkv.MkvShape(64, 8, 32768, 128, 0, None)
    assert mkv.mkv_workspace_size(shape, 0) > 32 << 20
    rc = mkv.load().mkv_compress_noalloc(None, None, shape, 0.5, None, 0, 0, 16384, None, None, None, None, None,
                                         None)
    assert rc == mkv.MKV_ERR_UNSUPPORTED
