"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle on
the same seeded inputs.  Routing, gate weights, grouping and the quantised
activations are compared bit for bit; the layer output within
rel-L2 <= 5e-3 and max-abs <= 3e-2 * rms(y_oracle), with the oracle routed
by the GPU's own fp32 logits."""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def h():
    import _harness
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import moe_expert_ffn_02_gb300 as moe
    moe.load()       # no fallback: the extension must be present
    return _harness


def small_wl(E, k, H=256, I=256, T=64, n_shared=1, zipf=0.0, name="small"):
    return synth.Workload(name, T, H, I, E, k, n_shared=n_shared, zipf_s=zipf)


# ------------------------------------------------------------------ routing

@pytest.mark.parametrize("E,k,T", [(8, 2, 64), (256, 8, 1), (256, 8, 16), (256, 8, 1000), (384, 8, 333),
                                   (1024, 32, 70), (5, 5, 7), (64, 6, 0)])
def test_route_from_logits_bit_exact(h, E, k, T):
    wl = small_wl(E, k, H=128, I=128, T=T)
    inp = synth.make_inputs(wl, seed=1)
    layer = h.make_layer(wl, inp)
    rng = np.random.default_rng(E + k + T)
    L = rng.normal(0, 1, (T, E)).astype(np.float32)
    if T > 3:
        L[0, :] = 0.75                            # all tied -> ids 0..k-1
        L[1, : E // 2] = np.float32(-0.5)         # partial ties
        L[2, 0], L[2, E - 1] = np.float32(-0.0), np.float32(0.0)
        L[3] = np.round(L[3] * 4) / 4             # many exact ties
    got = h.route_from_logits(layer, L)
    ref = oracle.route_from_logits(L, k)
    h.assert_routing_equal(got, ref)
    layer.close()


def test_router_logits_tolerance_and_routing(h):
    wl = synth.WORKLOADS["tiny"]
    inp = synth.make_inputs(wl, seed=0)
    layer = h.make_layer(wl, inp)
    got = h.route(layer, inp["x"])
    Lref = oracle.logits(inp["x"], inp["router_w"], inp["router_b"])
    assert np.all(np.abs(got["logits"] - Lref) <= 1e-5 * (1 + np.abs(Lref)))
    h.assert_routing_equal(got, oracle.route_from_logits(got["logits"], wl.top_k))
    h.count_routing_switches(got["topk_ids"], Lref, wl.top_k)
    layer.close()


# ------------------------------------------------------------------ layer, small shapes

def check_layer(h, wl, inp, mode, seed_rows=None):
    import moe_expert_ffn_02_gb300 as moe
    layer = h.make_layer(wl, inp)
    y, dbg = h.run_forward(layer, inp["x"], mode)
    r = h.route(layer, inp["x"])
    ref_route = oracle.route_from_logits(r["logits"], wl.top_k)
    h.assert_routing_equal(dbg, ref_route)
    xq, sx = oracle.quant_1x128(synth.bf16_to_f32(inp["x"]))
    assert np.array_equal(dbg["xq"], xq), "quantised x differs"
    assert np.array_equal(dbg["sx"].view(np.uint32), sx.view(np.uint32)), "x scales differ"
    rel, mx = h.check_layer_output(inp, wl.top_k, dbg, y)
    layer.close()
    return rel, mx, y


@pytest.mark.parametrize("mode", [1, 2])
def test_tiny_layer_parity(h, mode):
    wl = synth.WORKLOADS["tiny"]
    check_layer(h, wl, synth.make_inputs(wl, seed=0), mode)


@pytest.mark.parametrize("mode,T,k", [(1, 400, 8), (2, 64, 16)])
def test_many_experts_group_table_in_place(h, mode, T, k):
    """512 routed experts + shared, ~450-510 of them touched: more groups than
    the expert GEMMs copy into shared memory (385), so they decode their units
    from the table in place."""
    wl = small_wl(512, k, H=256, I=256, T=T)
    check_layer(h, wl, synth.make_inputs(wl, seed=8), mode)


@pytest.mark.parametrize("T", [1, 3, 17, 64])
def test_decode_entry_small_batches(h, T):
    wl = small_wl(16, 4, H=384, I=256, T=T)
    check_layer(h, wl, synth.make_inputs(wl, seed=5), 2)


@pytest.mark.parametrize("T,E,k,zipf,shared", [(300, 8, 2, 0.0, 1), (1000, 32, 4, 1.2, 1), (257, 16, 3, 0.0, 0),
                                               (129, 4, 4, 0.0, 1)])
def test_prefill_ragged_and_skewed(h, T, E, k, zipf, shared):
    """Several 64-row tiles per expert, ragged tails, empty experts (Zipf
    bias), no shared expert, and k = E (every token picks every expert)."""
    wl = small_wl(E, k, H=512, I=384, T=T, n_shared=shared, zipf=zipf)
    inp = synth.make_inputs(wl, seed=7)
    if zipf:
        inp["router_b"] = inp["router_b"] * 8.0     # push hard: some experts get no rows
    layer = h.make_layer(wl, inp)
    r = h.route(layer, inp["x"])
    layer.close()
    counts = np.diff(r["expert_offsets"])
    if zipf:
        assert counts.min() == 0 and counts.max() > 64
    check_layer(h, wl, inp, 1)


def test_zero_tokens_is_a_noop(h):
    import moe_expert_ffn_02_gb300 as moe
    wl = synth.WORKLOADS["tiny"]
    inp = synth.make_inputs(wl, seed=0)
    layer = h.make_layer(wl, inp)
    off = torch.full((wl.n_experts + 1,), 7, dtype=torch.int32, device="cuda")
    ws, nb = layer.workspace(0, moe.MODE_PREFILL)
    moe.moe_forward_prefill(layer.handle, 0, 0, 0, {"expert_offsets": off.data_ptr()}, ws, nb, layer.stream)
    torch.cuda.synchronize()
    assert not off.any()
    with pytest.raises(moe.MoeError):
        moe.moe_forward_decode(layer.handle, 0, 0, 0, None, ws, nb, layer.stream)
    layer.close()


def test_determinism_and_token_permutation(h):
    wl = small_wl(16, 4, H=384, I=256, T=200)
    inp = synth.make_inputs(wl, seed=9)
    layer = h.make_layer(wl, inp)
    y1, _ = h.run_forward(layer, inp["x"], 1, want_dbg=False)
    y2, _ = h.run_forward(layer, inp["x"], 1, want_dbg=False)
    assert np.array_equal(y1, y2)
    perm = np.random.default_rng(3).permutation(wl.T)
    yp, _ = h.run_forward(layer, inp["x"][perm], 1, want_dbg=False)
    assert np.array_equal(yp, y1[perm])
    # decode (16-token tiles, weights as the 128-row MMA operand) and prefill
    # (128-token tiles) compute the same function with different summation orders
    yd, _ = h.run_forward(layer, inp["x"][:64], 2, want_dbg=False)
    yq, _ = h.run_forward(layer, inp["x"][:64], 1, want_dbg=False)
    a, b = synth.bf16_to_f32(yd).astype(np.float64), synth.bf16_to_f32(yq).astype(np.float64)
    assert np.linalg.norm(a - b) / np.linalg.norm(b) <= h.REL_L2_TOL
    layer.close()


def test_host_entry_matches_device_entry(h):
    import moe_expert_ffn_02_gb300 as moe
    wl = small_wl(16, 4, H=384, I=256, T=50)
    inp = synth.make_inputs(wl, seed=11)
    layer = h.make_layer(wl, inp)
    xh = torch.from_numpy(inp["x"].view(np.int16)).pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    for mode in (1, 2):
        y_dev, _ = h.run_forward(layer, inp["x"], mode, want_dbg=False)
        ws, nb = layer.workspace(wl.T, mode)
        moe.moe_forward_host(layer.handle, mode, xh.data_ptr(), wl.T, yh.data_ptr(), ws, nb, layer.stream)
        assert np.array_equal(yh.numpy().view(np.uint16), y_dev)
    layer.close()


def test_profile_selects_stages_and_changes_no_result(h):
    """The measurement hook times every stage, or only the selected ones
    (the others read -1), and the layer output is the same either way."""
    import moe_expert_ffn_02_gb300 as moe
    wl = small_wl(16, 4, H=384, I=256, T=50)
    inp = synth.make_inputs(wl, seed=12)
    layer = h.make_layer(wl, inp)
    y0, _ = h.run_forward(layer, inp["x"], 2, want_dbg=False)
    for stages in (None, ("gate_up",), ("route", "down")):
        moe.moe_profile_enable(layer.handle, True, stages=stages)
        y1, _ = h.run_forward(layer, inp["x"], 2, want_dbg=False)
        ms = moe.moe_profile_read(layer.handle)
        timed = set(moe.PROFILE_STAGES if stages is None else stages)
        for name, v in ms.items():
            assert (v >= 0.0) if name in timed else (v == -1.0), (stages, ms)
        assert np.array_equal(y1, y0)
        moe.moe_profile_enable(layer.handle, False)
    for bad in (moe.PROFILE_SELECT, 7, moe.PROFILE_SELECT | 0x40):   # no stage; no selector; unknown stage
        with pytest.raises(moe.MoeError):
            moe._check(moe.load().moe_profile_enable(layer.handle, bad))
    layer.close()


def test_bounded_wait_reports_timeout_without_fault(h):
    import moe_expert_ffn_02_gb300 as moe
    wl = synth.WORKLOADS["tiny"]
    inp = synth.make_inputs(wl, seed=0)
    layer = h.make_layer(wl, inp)
    moe.moe_set_wait_limit(layer.handle, 2000)          # 2 ms
    moe.moe_debug_timeout_probe(layer.handle, layer.stream)
    st, flags = moe.moe_get_device_status(layer.handle, layer.stream)
    assert st == 6 and flags & moe.DEV_WAIT_TIMEOUT      # MOE_ERR_TIMEOUT
    st, flags = moe.moe_get_device_status(layer.handle, layer.stream)
    assert st == 0 and flags == 0                        # read-and-clear
    # the context is still usable
    moe.moe_set_wait_limit(layer.handle, 2_000_000)
    check_layer(h, wl, inp, 1)
    layer.close()


def _raw_forward(layer, x_bits, mode):
    """One forward call without the status assertion of run_forward."""
    import moe_expert_ffn_02_gb300 as moe
    T = x_bits.shape[0]
    x = torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).cuda()
    y = torch.zeros_like(x)
    ws, nb = layer.workspace(T, mode)
    fn = moe.moe_forward_prefill if mode == moe.MODE_PREFILL else moe.moe_forward_decode
    fn(layer.handle, x.data_ptr(), T, y.data_ptr(), None, ws, nb, layer.stream)
    st, flags = moe.moe_get_device_status(layer.handle, layer.stream)
    return st, flags, y.cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("mode,T", [(1, 200), (2, 16)])
def test_planted_faults_are_flagged_without_a_fault(h, mode, T):
    """Fault injection on the host side (moe_debug_inject): a routing id
    outside [0, E) planted between top-k and grouping, and an internal row
    outside the permuted buffers planted after grouping.  The kernels must
    flag each in the device word (MOE_ERR_DEVICE_CHECK with the fault's bit),
    clamp or skip it so nothing leaves the buffers, and the context must stay
    usable: the next clean call gives the clean output bit for bit."""
    import moe_expert_ffn_02_gb300 as moe
    wl = small_wl(16, 4, H=384, I=256, T=T)
    inp = synth.make_inputs(wl, seed=13)
    layer = h.make_layer(wl, inp)
    st, flags, y0 = _raw_forward(layer, inp["x"], mode)
    assert (st, flags) == (0, 0)
    for fault in (moe.DEV_BAD_EXPERT_ID, moe.DEV_BAD_ROW):
        moe.moe_debug_inject(layer.handle, fault)
        st, flags, _ = _raw_forward(layer, inp["x"], mode)
        assert st == 5 and flags == fault, (fault, st, flags)      # MOE_ERR_DEVICE_CHECK, that bit only
        st, flags, y1 = _raw_forward(layer, inp["x"], mode)          # fires once; the context is intact
        assert (st, flags) == (0, 0)
        assert np.array_equal(y1, y0)
    with pytest.raises(moe.MoeError):
        moe.moe_debug_inject(layer.handle, moe.DEV_WAIT_TIMEOUT)     # not a plantable fault
    layer.close()


def test_calls_on_another_device_are_rejected(h):
    """A handle records the device it was created on; a call made while
    another device is current is rejected before anything is enqueued.  With
    one GPU the mismatch is shown with a stand-in handle that records device
    7 (the handle's device field follows its 24-byte descriptor)."""
    import ctypes
    import moe_expert_ffn_02_gb300 as moe
    lib = moe.load()
    fake = (ctypes.c_int32 * 4096)()
    fake[6] = 7
    x = torch.zeros((8, 256), dtype=torch.int16, device="cuda")
    y = torch.full_like(x, 5)
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    calls = [
        lambda: lib.moe_forward_prefill(fake, x.data_ptr(), 8, y.data_ptr(), None, ws.data_ptr(), ws.numel(), None),
        lambda: lib.moe_forward_decode(fake, x.data_ptr(), 8, y.data_ptr(), None, ws.data_ptr(), ws.numel(), None),
        lambda: lib.moe_route(fake, x.data_ptr(), 8, None, ws.data_ptr(), ws.numel(), None),
        lambda: lib.moe_route_from_logits(fake, ws.data_ptr(), 8, None, ws.data_ptr(), ws.numel(), None),
        lambda: lib.moe_route_from_logits_noalloc(fake, ws.data_ptr(), 8, None, None),
        lambda: lib.moe_forward_host(fake, 1, 0x1000, 8, 0x1000, ws.data_ptr(), ws.numel(), None),
        lambda: lib.moe_tiles_load(fake, ws.data_ptr(), None),
        lambda: lib.moe_debug_timeout_probe(fake, None),
        lambda: lib.moe_profile_enable(fake, 1),
    ]
    for call in calls:
        assert call() == 1                                   # MOE_ERR_INVALID_ARG
        assert "is not the layer's device (7)" in moe.moe_last_error()
    torch.cuda.synchronize()
    assert bool((y == 5).all())


def test_argument_errors_enqueue_nothing(h):
    import moe_expert_ffn_02_gb300 as moe
    wl = synth.WORKLOADS["tiny"]
    inp = synth.make_inputs(wl, seed=0)
    layer = h.make_layer(wl, inp)
    ws, nb = layer.workspace(8, moe.MODE_PREFILL)
    x = torch.zeros((8, wl.hidden), dtype=torch.int16, device="cuda")
    y = torch.zeros_like(x)
    with pytest.raises(moe.MoeError) as e:
        moe.moe_forward_prefill(layer.handle, x.data_ptr(), 8, y.data_ptr(), None, ws, 1024, layer.stream)
    assert e.value.status == 3                           # MOE_ERR_WORKSPACE
    with pytest.raises(moe.MoeError) as e:
        moe.moe_forward_prefill(layer.handle, x.data_ptr() + 2, 8, y.data_ptr(), None, ws, nb, layer.stream)
    assert e.value.status == 1
    with pytest.raises(moe.MoeError) as e:
        moe.moe_forward_decode(layer.handle, x.data_ptr(), 65, y.data_ptr(), None, ws, nb, layer.stream)
    assert e.value.status == 2
    assert not y.any()
    layer.close()


# ------------------------------------------------------------------ full-size configurations

def group_edge_tokens(r):
    """The first and the last token of every expert's group: the rows at the
    boundaries of every group's first and last tile."""
    off, st = r["offsets"], r["sorted_token"]
    toks = set()
    for e in range(len(off) - 1):
        if off[e + 1] > off[e]:
            toks.add(int(st[off[e]]))
            toks.add(int(st[off[e + 1] - 1]))
    return toks


def sample_rows(T, r, n_rand, seed=0):
    """Tokens to check one by one: both ends of the batch, a seeded random
    subset of n_rand tokens, and the first and last token of every expert's
    group."""
    rng = np.random.default_rng(seed)
    rows = set(range(min(8, T))) | set(range(max(0, T - 8), T))
    rows |= set(rng.choice(T, size=min(n_rand, T), replace=False).tolist())
    rows |= group_edge_tokens(r)
    return np.array(sorted(rows), dtype=np.int32)


@pytest.mark.parametrize("name", ["ds_decode_t1", "ds_decode_t4", "ds_decode_t16"])
def test_deepseek_decode_layer(h, ds_inputs, name):
    wl = synth.WORKLOADS[name]
    base = ds_inputs
    inp = dict(base, x=synth.bf16_normal(0, synth.STREAM_X, (wl.T, wl.hidden)))
    layer = h.make_layer(wl, inp)
    y, dbg = h.run_forward(layer, inp["x"], 2)
    r = h.route(layer, inp["x"])
    Lref = oracle.logits(inp["x"], inp["router_w"], None)
    assert np.all(np.abs(r["logits"] - Lref) <= 1e-5 * (1 + np.abs(Lref)))
    ref_route = oracle.route_from_logits(r["logits"], wl.top_k)
    h.assert_routing_equal(dbg, ref_route)
    h.count_routing_switches(r["topk_ids"], Lref, wl.top_k)
    xq, sx = oracle.quant_1x128(synth.bf16_to_f32(inp["x"]))
    assert np.array_equal(dbg["xq"], xq) and np.array_equal(dbg["sx"], sx)
    h.check_layer_output(inp, wl.top_k, dbg, y)
    layer.close()


@pytest.fixture(scope="module")
def ds_inputs():
    wl = synth.WORKLOADS["ds_prefill_8k"]
    return synth.make_inputs(wl, seed=0)


def _prefill_full_size(h, wl, inp, n_rand):
    """The full-size prefill layer through the C ABI, routing checked bit for
    bit on every token, logits / quantised x / layer output on the tokens
    `rows` (every token when n_rand is None).  Returns what the caller needs
    for further checks."""
    layer = h.make_layer(wl, inp)
    y, dbg = h.run_forward(layer, inp["x"], 1)
    r = h.route(layer, inp["x"])
    ref_route = oracle.route_from_logits(r["logits"], wl.top_k)
    h.assert_routing_equal(dbg, ref_route)
    rows = None if n_rand is None else sample_rows(wl.T, ref_route, n_rand)
    sub = np.arange(wl.T) if rows is None else rows
    Lref = oracle.logits(inp["x"][sub], inp["router_w"], inp["router_b"])
    assert np.all(np.abs(r["logits"][sub] - Lref) <= 1e-5 * (1 + np.abs(Lref)))
    h.count_routing_switches(r["topk_ids"][sub], Lref, wl.top_k)
    xq, sx = oracle.quant_1x128(synth.bf16_to_f32(inp["x"][sub]))
    assert np.array_equal(dbg["xq"][sub], xq) and np.array_equal(dbg["sx"][sub], sx)
    h.check_layer_output(inp, wl.top_k, dbg, y, rows=rows)
    return layer, dbg, ref_route


def test_deepseek_prefill_8k_every_token(h, ds_inputs):
    """The 8K-token DeepSeek-V3 prefill layer, every one of its 8,192 tokens
    against the oracle (about 1.5 minutes of oracle time on 16 cores)."""
    wl = synth.WORKLOADS["ds_prefill_8k"]
    inp = dict(ds_inputs, x=synth.bf16_normal(0, synth.STREAM_X, (wl.T, wl.hidden)))
    layer, _, _ = _prefill_full_size(h, wl, inp, None)
    layer.close()


def _hottest(ref_route):
    counts = np.diff(ref_route["offsets"])
    return int(np.argmax(counts)), counts


def test_skewed_32k_prefill_subset_and_hottest_expert(h, ds_inputs):
    """The Zipf-skewed 32K layer: a seeded subset of 4,096 tokens plus the
    first and last token of every group against the whole-layer oracle, and
    every token routed to the hottest expert (about 32,000: every tile of
    the largest group) against that expert alone."""
    wl = synth.WORKLOADS["skew_32k"]
    inp = dict(ds_inputs, x=synth.bf16_normal(0, synth.STREAM_X, (wl.T, wl.hidden)), router_b=synth.router_bias(wl, 0))
    layer, dbg, ref_route = _prefill_full_size(h, wl, inp, 4096)
    hot, counts = _hottest(ref_route)
    mean = wl.T * wl.top_k / wl.n_experts
    assert counts.max() > 10 * mean and counts.min() == 0
    n = h.check_hot_expert(layer, inp, wl.top_k, dbg, inp["x"], 1, hot)
    assert n == counts[hot]
    layer.close()


def test_kimi_prefill_layer_subset_and_hottest_expert(h):
    """The Kimi-K2-shaped 64K layer (384 experts): a seeded subset of 4,096
    tokens plus every group's first and last token against the whole-layer
    oracle, and every token of the hottest expert against that expert."""
    wl = synth.WORKLOADS["kimi_64k"]
    inp = synth.make_inputs(wl, seed=0)
    layer, dbg, ref_route = _prefill_full_size(h, wl, inp, 4096)
    hot, counts = _hottest(ref_route)
    n = h.check_hot_expert(layer, inp, wl.top_k, dbg, inp["x"], 1, hot)
    assert n == counts[hot]
    layer.close()
