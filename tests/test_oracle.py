"""Pins for the CPU oracle: every check here compares it with something other
than itself (the FP8 format's closed form, an independent library routine,
brute force with a different loop structure, invariants, hand-computed
closed forms).  No GPU needed."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth


def torch_e4m3_decode(codes):
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def torch_e4m3_encode(v):
    return torch.from_numpy(np.asarray(v, dtype=np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


# ----------------------------------------------------------------------------- FP8 codec

def test_e4m3_decode_all_codes_closed_form():
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.e4m3_decode(codes)
    # closed form of the format: bias 7, exponent 0 subnormal, S.1111.111 NaN
    for c in range(256):
        s, e, m = c >> 7, (c >> 3) & 15, c & 7
        if e == 15 and m == 7:
            assert math.isnan(got[c])
            continue
        mag = (m / 8.0) * 2.0 ** -6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7)
        assert got[c] == (-mag if s else mag), c
    # landmarks of the format
    assert got[0x7E] == 448.0 and got[0xFE] == -448.0
    assert got[0x08] == 2.0 ** -6 and got[0x01] == 2.0 ** -9 and got[0x38] == 1.0
    # and an independent library decoder agrees on every finite code
    ref = torch_e4m3_decode(codes)
    fin = ~np.isnan(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.isnan(got), np.isnan(ref))


def test_e4m3_encode_roundtrip_midpoints_saturation():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = oracle.e4m3_decode(codes).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(vals), codes)
    pos = oracle.e4m3_decode(np.arange(127, dtype=np.uint8))
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)     # exact in fp32
    assert np.array_equal(mids.astype(np.float64), (pos[:-1] + pos[1:]) / 2)
    q = oracle.e4m3_encode(mids)
    lo = np.arange(126)
    expect = np.where(lo % 2 == 0, lo, lo + 1)                 # ties to the even code
    assert np.array_equal(q, expect.astype(np.uint8))
    # just above / below a midpoint
    assert np.array_equal(oracle.e4m3_encode(np.nextafter(mids, np.float32(np.inf))), (lo + 1).astype(np.uint8))
    assert np.array_equal(oracle.e4m3_encode(np.nextafter(mids, np.float32(0))), lo.astype(np.uint8))
    sat = oracle.e4m3_encode(np.array([448, 460, 464, 465, 1e6, -500, np.inf, -np.inf], dtype=np.float32))
    assert list(sat) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0x7E, 0xFE]
    assert oracle.e4m3_encode(np.array([np.nan], dtype=np.float32))[0] == 0x7F
    assert oracle.e4m3_encode(np.array([-0.0], dtype=np.float32))[0] == 0x80


def test_e4m3_encode_matches_library_in_range():
    rng = np.random.default_rng(1)
    v = np.concatenate([rng.normal(0, 50, 200000), rng.uniform(-463, 463, 50000),
                        rng.normal(0, 2 ** -7, 50000)]).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(v), torch_e4m3_encode(v))


# ----------------------------------------------------------------------------- exp32

def test_exp32_accuracy_and_special_values():
    x = np.linspace(-86.0, 0.0, 400001, dtype=np.float32)
    x = np.concatenate([x, -np.abs(np.random.default_rng(2).normal(0, 3, 200000)).astype(np.float32)])
    y = oracle.exp32(x).astype(np.float64)
    ref = np.exp(x.astype(np.float64))
    ulp = np.spacing(ref.astype(np.float32)).astype(np.float64)
    assert np.max(np.abs(y - ref) / ulp) <= 2.0
    assert oracle.exp32(np.float32([0.0]))[0] == 1.0
    assert oracle.exp32(np.float32([-86.5, -100.0, -np.inf]))[:].tolist() == [0.0, 0.0, 0.0]
    xs = np.sort(x)
    assert np.all(np.diff(oracle.exp32(xs)) >= 0)             # monotone


# ----------------------------------------------------------------------------- 1x128 quantisation

def test_quant_amax_maps_to_448_and_zero_group():
    rng = np.random.default_rng(3)
    v = rng.normal(0, 1, (16, 512)).astype(np.float32)
    v[3, 128:256] = 0.0
    q, s = oracle.quant_1x128(v)
    g = v.reshape(16, 4, 128)
    qg = q.reshape(16, 4, 128)
    amax = np.abs(g).max(-1)
    assert s[3, 1] == 1.0 and not qg[3, 1].any()
    nz = amax > 0
    assert np.array_equal(s[nz], (amax[nz] / np.float32(448.0)).astype(np.float32))
    arg = np.abs(g).argmax(-1)
    top = np.take_along_axis(qg, arg[..., None], -1)[..., 0]
    assert np.all((top[nz] & 0x7F) == 0x7E)


def test_quant_is_lossless_on_representable_groups():
    rng = np.random.default_rng(4)
    codes = rng.integers(0, 256, (8, 384)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x10
    codes[:, ::128] = 0x7E                                    # every group reaches 448
    j = rng.integers(-20, 5, (8, 3))
    scale = np.repeat(2.0 ** j, 128, axis=1)
    v = (oracle.e4m3_decode(codes) * scale).astype(np.float32)
    q, s = oracle.quant_1x128(v)
    # -0 codes come back as +0 only if the value is +0; compare values
    assert np.array_equal(oracle.e4m3_decode(q), oracle.e4m3_decode(codes))
    assert np.array_equal(s.astype(np.float64), 2.0 ** j)


def test_quant_matches_library_conversion_and_error_bound():
    rng = np.random.default_rng(5)
    v = (rng.normal(0, 1, (64, 1024)) * rng.lognormal(0, 2, (64, 1))).astype(np.float32)
    q, s = oracle.quant_1x128(v)
    ratio = (v.reshape(64, 8, 128) / s[..., None]).astype(np.float32)
    assert np.array_equal(q.reshape(64, 8, 128), torch_e4m3_encode(ratio))
    back = oracle.e4m3_decode(q).reshape(64, 8, 128) * s[..., None]
    # error at most half a step of the E4M3 grid at that magnitude (plus fp32 slack)
    a = np.abs(ratio.astype(np.float64))
    step = np.where(a < 2 ** -6, 2.0 ** -9, 2.0 ** (np.floor(np.log2(np.maximum(a, 2 ** -6))) - 3))
    err = np.abs(back - v.reshape(64, 8, 128)) / s[..., None]
    assert np.all(err <= 0.5 * step * (1 + 1e-6) + 1e-30)


# ----------------------------------------------------------------------------- logits

def test_logits_one_hot_and_library_matmul():
    rng = np.random.default_rng(6)
    H, E, T = 256, 16, 12
    W = rng.normal(0, 0.1, (E, H)).astype(np.float32)
    b = rng.normal(0, 1, E).astype(np.float32)
    x = np.zeros((T, H), dtype=np.uint16)
    for t in range(T):
        x[t, 7 * t] = 0x3F80                                  # bf16 1.0
    L = oracle.logits(x, W, b)
    for t in range(T):
        assert np.array_equal(L[t], (W[:, 7 * t].astype(np.float64) + b).astype(np.float32))
    xr = synth.bf16_normal(9, 1, (T, H))
    L = oracle.logits(xr, W, None)
    ref = (synth.bf16_to_f32(xr).astype(np.float64) @ W.astype(np.float64).T)
    assert np.all(np.abs(L - ref) <= np.spacing(np.abs(ref).astype(np.float32)))


# ----------------------------------------------------------------------------- routing

def brute_topk(L, k):
    T, E = L.shape
    ids = np.empty((T, k), dtype=np.int32)
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-float(L[t, e]), e))
        ids[t] = order[:k]
    return ids


@pytest.mark.parametrize("E,k", [(8, 2), (16, 4), (256, 8), (384, 8), (5, 5)])
def test_routing_topk_brute_force_and_weights(E, k):
    rng = np.random.default_rng(E * 31 + k)
    T = 97
    L = rng.normal(0, 1, (T, E)).astype(np.float32)
    L[0, :] = 0.5                                              # all tied
    L[1, : E // 2] = np.float32(0.25)                          # partial ties
    L[2, 0], L[2, -1] = np.float32(-0.0), np.float32(0.0)      # -0 == +0
    L[2, 1:-1] = -3.0
    r = oracle.route_from_logits(L, k)
    assert np.array_equal(r["ids"], brute_topk(L, k))
    assert list(r["ids"][0]) == list(range(k))
    if k in (2, 4, 8):
        assert np.all(r["w"][0] == np.float32(1.0 / k))
    if k >= 2:
        assert list(r["ids"][2][:2]) == [0, E - 1]
    # weights: a renormalised softmax (fp64 reference) within a few ulp; sum ~ 1
    sel = np.take_along_axis(L.astype(np.float64), r["ids"].astype(np.int64), 1)
    ref = np.exp(sel - sel[:, :1])
    ref /= ref.sum(1, keepdims=True)
    assert np.all(np.abs(r["w"] - ref) <= 4 * np.spacing(ref.astype(np.float32)) + 1e-45)
    assert np.all(np.abs(r["w"].astype(np.float64).sum(1) - 1.0) <= k * 2.0 ** -23)
    assert np.all(np.diff(r["w"], axis=1) <= 0)                # rank order = weight order


def test_permutation_invariants():
    rng = np.random.default_rng(11)
    T, E, k = 333, 64, 6
    L = rng.normal(0, 1, (T, E)).astype(np.float32)
    L[:, 5] += 10.0                                            # one expert every token picks
    L[:, 9] -= 50.0                                            # one expert never chosen
    r = oracle.route_from_logits(L, k)
    ids, off, st, inv = r["ids"], r["offsets"], r["sorted_token"], r["inv_row"]
    counts = np.bincount(ids.reshape(-1), minlength=E)
    assert counts.sum() == T * k and counts[9] == 0 and counts[5] == T
    assert off[0] == 0 and np.array_equal(np.diff(off), counts)
    for t in range(T):
        assert len(set(ids[t].tolist())) == k
        for j in range(k):
            row = inv[t, j]
            assert st[row] == t and off[ids[t, j]] <= row < off[ids[t, j] + 1]
    assert np.array_equal(np.sort(inv.reshape(-1)), np.arange(T * k))
    for e in range(E):
        seg = st[off[e]:off[e + 1]]
        assert np.all(np.diff(seg) > 0)                        # ascending tokens inside an expert
    assert np.array_equal(np.bincount(st, minlength=T), np.full(T, k))


# ----------------------------------------------------------------------------- layer

def dequant_blocks(q, s):
    """Independent dequantisation: library decoder x block multiplier."""
    d = torch_e4m3_decode(q)
    return d * np.repeat(np.repeat(s.astype(np.float64), 128, axis=-2), 128, axis=-1)


def swiglu_dense(x, wg, wu, wd):
    g = wg @ x
    u = wu @ x
    h = g / (1.0 + np.exp(-g)) * u
    return wd @ h


def test_layer_one_expert_top1_equals_dense_swiglu():
    wl = synth.Workload("one", 5, 256, 384, 1, 1, n_shared=0)
    inp = synth.make_inputs(wl, seed=3)
    for kname in ("sh_gate",):
        assert kname not in inp or wl.n_shared
    inp = {k: v for k, v in inp.items() if not k.startswith("sh")}
    ids = np.zeros((5, 1), dtype=np.int32)
    w = np.ones((5, 1), dtype=np.float32)
    y, y64 = oracle.forward(inp, 1, ids, w, exact_act=True, want_f64=True)
    wg = dequant_blocks(inp["w_gate"][0], inp["s_gate"][0])
    wu = dequant_blocks(inp["w_up"][0], inp["s_up"][0])
    wd = dequant_blocks(inp["w_down"][0], inp["s_down"][0])
    x = synth.bf16_to_f32(inp["x"]).astype(np.float64)
    ref = np.stack([swiglu_dense(x[t], wg, wu, wd) for t in range(5)])
    assert np.allclose(y64, ref, rtol=1e-12, atol=1e-15)
    # the routing step gives weight exactly 1 for a single selected expert
    r = oracle.route_from_logits(np.zeros((5, 1), np.float32), 1)
    assert np.all(r["w"] == 1.0)


def test_layer_brute_force_all_experts_exact_activations(tiny_inputs):
    wl, inp = tiny_inputs
    k = wl.top_k
    L = oracle.logits(inp["x"], inp["router_w"], inp["router_b"])
    r = oracle.route_from_logits(L, k)
    y, y64 = oracle.forward(inp, k, r["ids"], r["w"], exact_act=True, want_f64=True)
    x = synth.bf16_to_f32(inp["x"]).astype(np.float64)
    E = wl.n_experts
    per_expert = []
    for e in range(E):          # every expert on every token, then select
        wg = dequant_blocks(inp["w_gate"][e], inp["s_gate"][e])
        wu = dequant_blocks(inp["w_up"][e], inp["s_up"][e])
        wd = dequant_blocks(inp["w_down"][e], inp["s_down"][e])
        G, U = x @ wg.T, x @ wu.T
        per_expert.append((G / (1 + np.exp(-G)) * U) @ wd.T)
    per_expert = np.stack(per_expert)                          # [E][T][H]
    sg = dequant_blocks(inp["sh_gate"][0], inp["sh_s_gate"][0])
    su = dequant_blocks(inp["sh_up"][0], inp["sh_s_up"][0])
    sd = dequant_blocks(inp["sh_down"][0], inp["sh_s_down"][0])
    G, U = x @ sg.T, x @ su.T
    ref = (G / (1 + np.exp(-G)) * U) @ sd.T
    for j in range(k):
        ref = ref + r["w"][:, j:j + 1].astype(np.float64) * per_expert[r["ids"][:, j], np.arange(wl.T)]
    assert np.allclose(y64, ref, rtol=1e-11, atol=1e-14)
    yb = synth.bf16_to_f32(y).astype(np.float64)
    assert np.all(np.abs(yb - ref) <= np.spacing(np.abs(ref).astype(np.float32)) * 2 ** 16 / 2 + 1e-30)


def test_layer_brute_force_quantised_activations(tiny_inputs):
    """Same brute force with the (separately pinned) 1x128 quantiser applied to x and h."""
    wl, inp = tiny_inputs
    k = wl.top_k
    L = oracle.logits(inp["x"], inp["router_w"], inp["router_b"])
    r = oracle.route_from_logits(L, k)
    _, y64 = oracle.forward(inp, k, r["ids"], r["w"], want_f64=True)
    xf = synth.bf16_to_f32(inp["x"])
    xq, sx = oracle.quant_1x128(xf)
    xd = oracle.e4m3_decode(xq) * np.repeat(sx.astype(np.float64), 128, axis=1)

    def ffn(wg, wu, wd):
        G, U = xd @ wg.T, xd @ wu.T
        h32 = (G / (1 + np.exp(-G)) * U).astype(np.float32)
        hq, sh = oracle.quant_1x128(h32)
        hd = oracle.e4m3_decode(hq) * np.repeat(sh.astype(np.float64), 128, axis=1)
        return hd @ wd.T

    ref = ffn(dequant_blocks(inp["sh_gate"][0], inp["sh_s_gate"][0]),
              dequant_blocks(inp["sh_up"][0], inp["sh_s_up"][0]),
              dequant_blocks(inp["sh_down"][0], inp["sh_s_down"][0]))
    outs = [ffn(dequant_blocks(inp["w_gate"][e], inp["s_gate"][e]), dequant_blocks(inp["w_up"][e], inp["s_up"][e]),
                dequant_blocks(inp["w_down"][e], inp["s_down"][e])) for e in range(wl.n_experts)]
    for j in range(k):
        sel = np.stack([outs[r["ids"][t, j]][t] for t in range(wl.T)])
        ref = ref + r["w"][:, j:j + 1].astype(np.float64) * sel
    # h is rounded to fp32 on both sides from fp64 values summed in different
    # orders; a rare 1-ulp difference can flip one h code, hence a loose bound
    rel = np.linalg.norm(y64 - ref) / np.linalg.norm(ref)
    assert rel < 1e-6
    assert np.mean(np.isclose(y64, ref, rtol=1e-12, atol=1e-15)) > 0.99


def test_layer_closed_form_single_weights():
    """Hand-computable case: one nonzero code per matrix, one-hot input."""
    H = I = 128
    wg = np.zeros((1, I, H), np.uint8); wu = np.zeros((1, I, H), np.uint8); wd = np.zeros((1, H, I), np.uint8)
    wg[0, 0, 0] = 0x38    # 1.0
    wu[0, 0, 0] = 0x40    # 2.0
    wd[0, 0, 0] = 0x38    # 1.0
    wd[0, 5, 0] = 0xC4    # -3.0
    inp = {"x": np.zeros((1, H), np.uint16), "w_gate": wg, "w_up": wu, "w_down": wd,
           "s_gate": np.full((1, 1, 1), 0.5, np.float32), "s_up": np.full((1, 1, 1), 0.25, np.float32),
           "s_down": np.full((1, 1, 1), 4.0, np.float32)}
    inp["x"][0, 0] = 0x4000                                   # bf16 2.0
    ids, w = np.zeros((1, 1), np.int32), np.ones((1, 1), np.float32)
    _, y64 = oracle.forward(inp, 1, ids, w, exact_act=True, want_f64=True)
    g = 1.0 * 0.5 * 2.0
    u = 2.0 * 0.25 * 2.0
    h = g / (1 + math.exp(-g)) * u
    assert y64[0, 0] == 4.0 * h and y64[0, 5] == -12.0 * h and np.count_nonzero(y64) == 2
    # quantised: x's group has amax 2 -> s = fp32(2/448), code 0x7E, value 448*s
    y, y64q = oracle.forward(inp, 1, ids, w, want_f64=True)
    sx = float(np.float32(2.0) / np.float32(448.0))
    a = 448.0 * sx
    g = 1.0 * 0.5 * a
    u = 2.0 * 0.25 * a
    h32 = float(np.float32(g / (1 + math.exp(-g)) * u))
    sh = float(np.float32(h32) / np.float32(448.0))
    hd = 448.0 * sh                                           # h is the group's amax -> code 0x7E
    assert y64q[0, 0] == 4.0 * hd and y64q[0, 5] == -12.0 * hd
    assert synth.bf16_to_f32(y)[0, 0] == np.float32(torch.tensor(4.0 * hd, dtype=torch.float64).to(torch.bfloat16).float().item())


def test_layer_invariances(tiny_inputs):
    wl, inp = tiny_inputs
    k = wl.top_k
    L = oracle.logits(inp["x"], inp["router_w"], inp["router_b"])
    r = oracle.route_from_logits(L, k)
    y = oracle.forward(inp, k, r["ids"], r["w"])
    # token permutation equivariance (bitwise)
    perm = np.random.default_rng(0).permutation(wl.T)
    inp_p = dict(inp, x=inp["x"][perm])
    y_p = oracle.forward(inp_p, k, r["ids"][perm], r["w"][perm])
    assert np.array_equal(y_p, y[perm])
    # expert relabelling equivariance (bitwise)
    rel = np.random.default_rng(1).permutation(wl.n_experts)     # new index of old expert e is rel[e]
    inv = np.argsort(rel)
    inp_r = dict(inp)
    for n in ("w_gate", "w_up", "w_down", "s_gate", "s_up", "s_down"):
        inp_r[n] = inp[n][inv]
    y_r = oracle.forward(inp_r, k, rel[r["ids"]].astype(np.int32), r["w"])
    assert np.array_equal(y_r, y)
    # routing from relabelled router rows selects the relabelled experts
    L_r = oracle.logits(inp["x"], inp["router_w"][inv], None)
    assert np.array_equal(L_r, L[:, inv])
    # doubling every down-projection multiplier doubles y exactly
    inp_d = dict(inp, s_down=inp["s_down"] * 2, sh_s_down=inp["sh_s_down"] * 2)
    _, y64 = oracle.forward(inp, k, r["ids"], r["w"], want_f64=True)
    _, y64d = oracle.forward(inp_d, k, r["ids"], r["w"], want_f64=True)
    assert np.array_equal(y64d, 2 * y64)
    # zero input -> zero output
    y0 = oracle.forward(dict(inp, x=np.zeros_like(inp["x"])), k, r["ids"], r["w"])
    assert not np.any(synth.bf16_to_f32(y0))
    # a token subset is evaluated exactly as in the full run
    rows = np.array([5, 0, 63, 17], dtype=np.int32)
    assert np.array_equal(oracle.forward(inp, k, r["ids"], r["w"], rows=rows), y[rows])


def test_oracle_thread_count_does_not_change_results(tiny_inputs):
    wl, inp = tiny_inputs
    L1 = oracle.logits(inp["x"], inp["router_w"], None, n_threads=1)
    L4 = oracle.logits(inp["x"], inp["router_w"], None, n_threads=4)
    assert np.array_equal(L1, L4)
    r = oracle.route_from_logits(L1, wl.top_k)
    assert np.array_equal(oracle.forward(inp, wl.top_k, r["ids"], r["w"], n_threads=1),
                          oracle.forward(inp, wl.top_k, r["ids"], r["w"], n_threads=3))


def test_h_override_with_own_codes_is_identity_and_one_code_is_closed_form(tiny_inputs):
    """The h-code override feeds given codes to the down projection: with the
    oracle's own codes nothing changes; changing one code of one (token,
    slot) moves y by exactly w * Wd[:, i] * (new - old) * s_block."""
    wl, inp = tiny_inputs
    k = wl.top_k
    L = oracle.logits(inp["x"], inp["router_w"], inp["router_b"])
    r = oracle.route_from_logits(L, k)
    y, y64, hrec = oracle.forward(inp, k, r["ids"], r["w"], want_f64=True, want_h=True)
    assert hrec["hq"].shape == (wl.T, k + 1, wl.inter)
    # the recorded codes are the 1x128 quantisation of the recorded fp32 h
    q, s = oracle.quant_1x128(hrec["h32"])
    assert np.array_equal(q, hrec["hq"]) and np.array_equal(s, hrec["sh"])
    y2, y64b = oracle.forward(inp, k, r["ids"], r["w"], want_f64=True, hq_in=hrec["hq"], sh_in=hrec["sh"])
    assert np.array_equal(y64b, y64) and np.array_equal(y2, y)
    t, j, i = 5, 1, 77                                        # token 5, routed slot 1, channel 77
    hq = hrec["hq"].copy()
    old = hq[t, j, i]
    new = old + 1 if (old & 0x7F) < 0x7E else old - 1
    hq[t, j, i] = new
    _, y64c = oracle.forward(inp, k, r["ids"], r["w"], want_f64=True, hq_in=hq, sh_in=hrec["sh"])
    e = r["ids"][t, j]
    wd_col = oracle.e4m3_decode(inp["w_down"][e][:, i]) * np.repeat(inp["s_down"][e][:, i // 128].astype(np.float64), 128)
    delta = (oracle.e4m3_decode(np.uint8(new)) - oracle.e4m3_decode(np.uint8(old))) * float(hrec["sh"][t, j, i // 128])
    expect = float(r["w"][t, j]) * wd_col * delta
    assert np.allclose(y64c[t] - y64[t], expect, rtol=1e-9, atol=1e-15)
    others = np.arange(wl.T) != t
    assert np.array_equal(y64c[others], y64[others])
