"""The layer's composition variants on the GPU, against the oracle.

- moe_forward_layers / LayerStackGraph: a stack of layers, each layer's output
  the next one's input, as one call and as one replayed CUDA graph (the
  decode step of the "LLM serving on heterogeneous hardware" lecture, section
  4.3).  Must equal the layers run one call at a time, bit for bit, and each
  layer must match the oracle on its own input.
- moe_forward_smallep: the SmallEP combine (partial sums of contiguous expert
  groups, reduced in rank order; CPU-GPU hybrid inference article, SmallEP
  section).  One rank is the plain combine bit for bit; more ranks stay
  within the layer tolerance.
- moe_forward_deferred: deferred slots split off into y_next (lecture section
  4.3, expert deferral); checked against the oracle's fp64 partial sums.
- Host-tile layers (moe_create_ex with MOE_CREATE_HOST_TILES) run through the
  two-slot ring of StreamedStack (the hybrid-inference article's
  Stream-Loading Prefill): must equal the same layers kept in HBM, bit for
  bit, and each layer must match the oracle on its own input.
"""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

REL, MAXABS = 5e-3, 3e-2


@pytest.fixture(scope="module")
def h():
    import _harness
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import moe_expert_ffn_02_gb300 as moe
    moe.load()       # no fallback: the extension must be present
    return _harness


def small_wl(E, k, H=256, I=256, T=64, n_shared=1):
    return synth.Workload("small", T, H, I, E, k, n_shared=n_shared)


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def bf16_f64(bits):
    return synth.bf16_to_f32(bits).astype(np.float64)


def close(y_bits, ref64, what):
    a, b = bf16_f64(y_bits), ref64
    rms = np.sqrt(np.mean(b * b))
    rel = np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30)
    mx = np.max(np.abs(a - b)) / max(rms, 1e-30) if a.size else 0.0
    print(f"[{what}] rel_l2={rel:.3e} max_abs/rms={mx:.3e}")
    assert rel <= REL and mx <= MAXABS, f"{what}: rel {rel:.3e}, max-abs {mx:.3e}"


# ------------------------------------------------------------------ layer stack

@pytest.mark.parametrize("mode,T", [(2, 16), (1, 200)])
def test_layer_stack_equals_single_calls_and_oracle(h, mode, T):
    import moe_expert_ffn_02_gb300 as moe
    wl = small_wl(8, 2, T=T)
    inps = [synth.make_inputs(wl, seed=s) for s in (1, 2, 3)]
    layers = [h.make_layer(wl, inp) for inp in inps]
    x0 = inps[0]["x"]

    # one call at a time, each layer checked against the oracle on its own input
    x = x0
    for l, (layer, inp) in enumerate(zip(layers, inps)):
        y, dbg = h.run_forward(layer, x, mode)
        inp_l = dict(inp, x=x)
        h.check_layer_output(inp_l, wl.top_k, dbg, y)
        x = y
    y_seq = x

    handles = [ly.handle for ly in layers]
    xd = dev(x0.view(np.int16))
    yd = torch.empty_like(xd)
    need = moe.moe_layers_workspace_bytes(handles, T, mode)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    moe.moe_forward_layers(handles, mode, xd.data_ptr(), T, yd.data_ptr(), ws.data_ptr(), need,
                           torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert np.array_equal(yd.cpu().numpy().view(np.uint16), y_seq)

    # captured once, replayed on new input
    xg = dev(x0.view(np.int16))
    yg = torch.empty_like(xg)
    g = moe.LayerStackGraph(handles, mode, xg, yg)
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(yg.cpu().numpy().view(np.uint16), y_seq)
    x1 = synth.make_inputs(wl, seed=9, with_experts=False)["x"]
    xg.copy_(dev(x1.view(np.int16)))
    g.replay()
    torch.cuda.synchronize()
    x = x1
    for layer in layers:
        x, _ = h.run_forward(layer, x, mode, want_dbg=False)
    assert np.array_equal(yg.cpu().numpy().view(np.uint16), x)
    for ly in layers:
        ly.close()


def test_layer_stack_argument_errors(h):
    import moe_expert_ffn_02_gb300 as moe
    wl = small_wl(8, 2, T=8)
    a = h.make_layer(wl, synth.make_inputs(wl, seed=1))
    wl2 = small_wl(8, 2, H=384, T=8)
    b = h.make_layer(wl2, synth.make_inputs(wl2, seed=1))
    with pytest.raises(moe.MoeError):
        moe.moe_layers_workspace_bytes([a.handle, b.handle], 8, 2)      # hidden sizes differ
    with pytest.raises(moe.MoeError):
        moe.moe_layers_workspace_bytes([a.handle], 65, 2)               # decode T > 64
    with pytest.raises(moe.MoeError):
        moe.moe_forward_layers([a.handle], 2, 0, 8, 0, 0, 0)             # no workspace
    a.close()
    b.close()


# ------------------------------------------------------------------ SmallEP

def _smallep(h, layer, x_bits, mode, n_ranks):
    import moe_expert_ffn_02_gb300 as moe
    T = x_bits.shape[0]
    x = dev(x_bits.view(np.int16))
    y = torch.empty_like(x)
    ws, nb = layer.workspace(T, mode)
    moe.moe_forward_smallep(layer.handle, mode, n_ranks, x.data_ptr(), T, y.data_ptr(), ws, nb, layer.stream)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(layer.handle, layer.stream) == (0, 0)
    return y.cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("mode,T,E,k", [(1, 300, 16, 4), (2, 16, 16, 4), (1, 129, 7, 7)])
def test_smallep_combine(h, mode, T, E, k):
    wl = small_wl(E, k, H=384, T=T)
    inp = synth.make_inputs(wl, seed=4)
    layer = h.make_layer(wl, inp)
    y, dbg = h.run_forward(layer, inp["x"], mode)
    assert np.array_equal(_smallep(h, layer, inp["x"], mode, 1), y), "one rank must be the plain combine"
    for P in (2, 3, E):
        yp = _smallep(h, layer, inp["x"], mode, P)
        assert np.array_equal(yp, _smallep(h, layer, inp["x"], mode, P)), "not deterministic"
        h.check_layer_output(inp, k, dbg, yp)
    layer.close()


def test_smallep_rejects_bad_rank_count(h):
    import moe_expert_ffn_02_gb300 as moe
    wl = small_wl(8, 2, T=8)
    layer = h.make_layer(wl, synth.make_inputs(wl, seed=1))
    ws, nb = layer.workspace(8, 2)
    for P in (0, 9):
        with pytest.raises(moe.MoeError):
            moe.moe_forward_smallep(layer.handle, 2, P, 0, 8, 0, ws, nb, layer.stream)
    layer.close()


# ------------------------------------------------------------------ deferral

def _deferred(h, layer, x_bits, mode, mask):
    import moe_expert_ffn_02_gb300 as moe
    T = x_bits.shape[0]
    x = dev(x_bits.view(np.int16))
    y_now, y_next = torch.empty_like(x), torch.empty_like(x)
    m = dev(mask.astype(np.uint8))
    ws, nb = layer.workspace(T, mode)
    moe.moe_forward_deferred(layer.handle, mode, x.data_ptr(), T, m.data_ptr(), y_now.data_ptr(), y_next.data_ptr(),
                             ws, nb, layer.stream)
    torch.cuda.synchronize()
    assert moe.moe_get_device_status(layer.handle, layer.stream) == (0, 0)
    return y_now.cpu().numpy().view(np.uint16), y_next.cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("mode,T", [(2, 32), (1, 200)])
def test_deferral_split(h, mode, T):
    E, k = 16, 4
    wl = small_wl(E, k, H=384, T=T)
    inp = synth.make_inputs(wl, seed=6)
    layer = h.make_layer(wl, inp)
    y, dbg = h.run_forward(layer, inp["x"], mode)

    now, nxt = _deferred(h, layer, inp["x"], mode, np.zeros((T, k), np.uint8))
    assert np.array_equal(now, y), "nothing deferred: y_now must be the plain output"
    assert not np.any(synth.bf16_to_f32(nxt)), "nothing deferred: y_next must be zero"

    rng = np.random.default_rng(T)
    mask = (rng.random((T, k)) < 0.4).astype(np.uint8)
    mask[:, :2] = 0                              # keep two undeferred slots per token
    now, nxt = _deferred(h, layer, inp["x"], mode, mask)
    ids, w = dbg["topk_ids"], dbg["topk_w"]
    kw = dict(hq_in=dbg["hq"], sh_in=dbg["sh"], want_f64=True)
    _, y_keep = oracle.forward(inp, k, ids, np.where(mask, 0.0, w).astype(np.float32), **kw)
    _, y_def = oracle.forward(inp, k, ids, np.where(mask, w, 0.0).astype(np.float32), **kw)
    _, y_sh = oracle.forward(inp, k, ids, np.zeros_like(w), **kw)
    close(now, y_keep, "y_now")
    close(nxt, y_def - y_sh, "y_next")
    layer.close()


# ------------------------------------------------------------------ host tiles, two-slot ring

@pytest.mark.parametrize("mode,T", [(1, 200), (2, 16)])
def test_streamed_stack_equals_resident(h, mode, T):
    import moe_expert_ffn_02_gb300 as moe
    wl = small_wl(8, 2, T=T)
    inps = [synth.make_inputs(wl, seed=s) for s in (11, 12, 13)]
    resident = [h.make_layer(wl, inp) for inp in inps]
    hosted = [h.make_layer(wl, inp, host_tiles=True) for inp in inps]
    x0 = dev(inps[0]["x"].view(np.int16))

    y_ref = torch.empty_like(x0)
    handles = [ly.handle for ly in resident]
    need = moe.moe_layers_workspace_bytes(handles, T, mode)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    moe.moe_forward_layers(handles, mode, x0.data_ptr(), T, y_ref.data_ptr(), ws.data_ptr(), need,
                           torch.cuda.current_stream().cuda_stream)

    y = torch.empty_like(x0)
    ring = moe.StreamedStack(hosted, mode, x0, y)
    for _ in range(2):                                  # a second pass reuses both slots
        y.zero_()
        ring.run()
        torch.cuda.synchronize()
        assert np.array_equal(y.cpu().numpy(), y_ref.cpu().numpy())
    for ly in hosted:
        assert moe.moe_get_device_status(ly.handle, 0) == (0, 0)

    # each host-tile layer alone (a one-layer ring) against the oracle on its own input, routed by the
    # GPU's fp32 logits (moe_route works on host-tile layers); the chain of one-layer rings must give the
    # three-layer ring's output bit for bit
    x_l = x0
    for ly, inp in zip(hosted, inps):
        y_l = torch.empty_like(x_l)
        moe.StreamedStack([ly], mode, x_l, y_l).run()
        torch.cuda.synchronize()
        xb = x_l.cpu().numpy().view(np.uint16)
        r = h.route(ly, xb)
        ref_route = oracle.route_from_logits(r["logits"], wl.top_k)
        assert np.array_equal(r["topk_ids"], ref_route["ids"])
        assert np.array_equal(r["topk_w"].view(np.uint32), ref_route["w"].view(np.uint32))
        _, y64 = oracle.forward(dict(inp, x=xb), wl.top_k, ref_route["ids"], ref_route["w"], want_f64=True)
        close(y_l.cpu().numpy().view(np.uint16), y64, f"streamed layer, mode {mode}")
        x_l = y_l
    assert np.array_equal(x_l.cpu().numpy(), y_ref.cpu().numpy())

    # a host-tile layer needs a slot; a resident layer has nothing to load
    ws1, nb1 = hosted[0].workspace(T, mode)
    with pytest.raises(moe.MoeError):
        moe.moe_forward_prefill(hosted[0].handle, x0.data_ptr(), T, y.data_ptr(), None, ws1, nb1, 0)
    with pytest.raises(moe.MoeError):
        moe.moe_tiles_load(resident[0].handle, ring.slots[0].data_ptr(), 0)
    assert moe.moe_tiles_bytes(hosted[0].handle) == moe.moe_tiles_bytes(resident[0].handle)
    for ly in resident + hosted:
        ly.close()
