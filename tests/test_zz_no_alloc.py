"""The allocation-free routing entry point, moe_route_from_logits_noalloc,
against the workspace entry point, moe_route_from_logits, through the C ABI.

The no-allocation variant is for callers that cannot allocate device memory
when they route (serving runtimes that give all of HBM to their own pools at
start-up, plain C callers without an allocator): its scratch is an array
built into the library.  Both entry points compute with the same device
functions (for decode-sized batches the workspace entry fuses them into one
kernel), so their results must agree bit for bit.  This file is collected last so that a run
that stops at the first failure has already run every other test."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _routing_buffers(T, E, k):
    return {
        "topk_ids": torch.full((T, k), -7, dtype=torch.int32, device="cuda"),
        "topk_w": torch.full((T, k), -7.0, dtype=torch.float32, device="cuda"),
        "expert_offsets": torch.full((E + 1,), -7, dtype=torch.int32, device="cuda"),
        "sorted_token": torch.full((max(T * k, 1),), -7, dtype=torch.int32, device="cuda"),
        "inv_row": torch.full((T, k), -7, dtype=torch.int32, device="cuda"),
    }


@pytest.mark.parametrize("E,sizes", [(256, (1000, 3000)), (256, (1, 16, 64)), (640, (64, 200))])
def test_noalloc_routing_matches_workspace_routing_on_two_calls(E, sizes):
    """Calls in a row of different sizes.  Decode-sized batches (T <= 64 with
    E <= 512) take the workspace entry's fused one-CTA routing kernel, while
    this entry runs the stages one by one; E = 640 takes the multi-kernel
    path on both sides."""
    import synth
    import moe_expert_ffn_02_gb300 as moe
    import _harness as h

    assert torch.cuda.is_available()
    moe.load()
    wl = synth.Workload("route", 64, 128, 128, E, 8)
    layer = h.make_layer(wl, synth.make_inputs(wl, seed=4))
    E, k = wl.n_experts, wl.top_k
    rng = np.random.default_rng(42 + E + sizes[0])
    for call, T in enumerate(sizes):                    # calls in a row, different sizes
        L = rng.normal(0, 1, (T, E)).astype(np.float32)
        L[0, :] = 0.5                                     # ties -> lowest indices
        if T > 1:
            L[1] = np.round(L[1] * 2) / 2
        Ld = torch.from_numpy(L).cuda()
        ref = _routing_buffers(T, E, k)
        ws, nbytes = layer.workspace(T, moe.MODE_ROUTE)
        moe.moe_route_from_logits(layer.handle, Ld.data_ptr(), T, {n: t.data_ptr() for n, t in ref.items()},
                                  ws, nbytes, layer.stream)
        got = _routing_buffers(T, E, k)
        moe.moe_route_from_logits_noalloc(layer.handle, Ld.data_ptr(), T, {n: t.data_ptr() for n, t in got.items()},
                                          layer.stream)
        torch.cuda.synchronize()
        for n in ref:
            a, b = got[n].cpu().numpy(), ref[n].cpu().numpy()
            assert np.array_equal(a.view(np.uint32), b.view(np.uint32)), f"call {call}: {n} differs"
        st, flags = moe.moe_get_device_status(layer.handle, layer.stream)
        assert st == 0 and flags == 0

    if E != 256 or sizes[0] != 1000:
        layer.close()
        return
    # beyond the built-in scratch: rejected before anything runs
    T = 40000
    Ld = torch.zeros((T, E), dtype=torch.float32, device="cuda")
    got = _routing_buffers(T, E, k)
    with pytest.raises(moe.MoeError) as e:
        moe.moe_route_from_logits_noalloc(layer.handle, Ld.data_ptr(), T, {n: t.data_ptr() for n, t in got.items()},
                                          layer.stream)
    assert e.value.status == 2                             # MOE_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert bool((got["topk_ids"] == -7).all())
    layer.close()
