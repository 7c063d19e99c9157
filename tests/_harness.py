"""Shared helpers for the GPU tests: upload seeded inputs, run the library
through its C ABI, and compare with the CPU oracle."""
from __future__ import annotations

import numpy as np
import torch

import moe_expert_ffn_02_gb300 as moe
import oracle
import synth

WEIGHT_KEYS = ("router_w", "router_b", "w_gate", "w_up", "w_down", "s_gate", "s_up", "s_down",
               "sh_gate", "sh_up", "sh_down", "sh_s_gate", "sh_s_up", "sh_s_down")


def to_dev(a):
    if a is None:
        return None
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def make_layer(wl: synth.Workload, inp: dict, host_tiles: bool = False) -> moe.Layer:
    dev = {k: to_dev(inp.get(k)) for k in WEIGHT_KEYS}
    layer = moe.Layer(wl.hidden, wl.inter, wl.n_experts, wl.top_k, dev, n_shared=wl.n_shared, host_tiles=host_tiles)
    del dev
    return layer


def run_forward(layer: moe.Layer, x_bits: np.ndarray, mode: int, want_dbg: bool = True):
    """x_bits: uint16 [T][H].  Returns (y uint16 [T][H], dbg dict of numpy)."""
    T, H = x_bits.shape
    E, k = layer.desc.n_experts, layer.desc.top_k
    x = to_dev(x_bits.view(np.int16))
    y = torch.empty((T, H), dtype=torch.int16, device="cuda")
    dbg = None
    bufs = {}
    if want_dbg:
        bufs = {
            "topk_ids": torch.empty((T, k), dtype=torch.int32, device="cuda"),
            "topk_w": torch.empty((T, k), dtype=torch.float32, device="cuda"),
            "expert_offsets": torch.empty((E + 1,), dtype=torch.int32, device="cuda"),
            "sorted_token": torch.empty((max(T * k, 1),), dtype=torch.int32, device="cuda"),
            "inv_row": torch.empty((T, k), dtype=torch.int32, device="cuda"),
            "xq": torch.empty((T, H), dtype=torch.uint8, device="cuda"),
            "sx": torch.empty((T, H // 128), dtype=torch.float32, device="cuda"),
        }
        S = k + layer.desc.n_shared
        I = layer.desc.inter
        bufs["hq"] = torch.empty((T, S, I), dtype=torch.uint8, device="cuda")
        bufs["sh"] = torch.empty((T, S, I // 128), dtype=torch.float32, device="cuda")
        dbg = {n: t.data_ptr() for n, t in bufs.items()}
    ws, nbytes = layer.workspace(T, mode)
    fn = moe.moe_forward_prefill if mode == moe.MODE_PREFILL else moe.moe_forward_decode
    fn(layer.handle, x.data_ptr() if T else 0, T, y.data_ptr() if T else 0, dbg, ws, nbytes, layer.stream)
    torch.cuda.synchronize()
    st, flags = moe.moe_get_device_status(layer.handle, layer.stream)
    assert st == 0 and flags == 0, f"device status {st} flags {flags:#x}"
    out = {n: t.cpu().numpy() for n, t in bufs.items()}
    if "sorted_token" in out:
        out["sorted_token"] = out["sorted_token"][: T * k]
    return y.cpu().numpy().view(np.uint16), out


def route(layer: moe.Layer, x_bits: np.ndarray):
    """moe_route: logits and routing outputs as numpy."""
    T, H = x_bits.shape
    E, k = layer.desc.n_experts, layer.desc.top_k
    x = to_dev(x_bits.view(np.int16))
    bufs = {
        "logits": torch.empty((T, E), dtype=torch.float32, device="cuda"),
        "topk_ids": torch.empty((T, k), dtype=torch.int32, device="cuda"),
        "topk_w": torch.empty((T, k), dtype=torch.float32, device="cuda"),
        "expert_offsets": torch.empty((E + 1,), dtype=torch.int32, device="cuda"),
        "sorted_token": torch.empty((max(T * k, 1),), dtype=torch.int32, device="cuda"),
        "inv_row": torch.empty((T, k), dtype=torch.int32, device="cuda"),
    }
    ws, nbytes = layer.workspace(T, moe.MODE_ROUTE)
    moe.moe_route(layer.handle, x.data_ptr() if T else 0, T, {n: t.data_ptr() for n, t in bufs.items()}, ws, nbytes,
                  layer.stream)
    torch.cuda.synchronize()
    out = {n: t.cpu().numpy() for n, t in bufs.items()}
    out["sorted_token"] = out["sorted_token"][: T * k]
    return out


def route_from_logits(layer: moe.Layer, L: np.ndarray):
    T = L.shape[0]
    E, k = layer.desc.n_experts, layer.desc.top_k
    Ld = to_dev(L.astype(np.float32))
    bufs = {
        "topk_ids": torch.empty((T, k), dtype=torch.int32, device="cuda"),
        "topk_w": torch.empty((T, k), dtype=torch.float32, device="cuda"),
        "expert_offsets": torch.empty((E + 1,), dtype=torch.int32, device="cuda"),
        "sorted_token": torch.empty((max(T * k, 1),), dtype=torch.int32, device="cuda"),
        "inv_row": torch.empty((T, k), dtype=torch.int32, device="cuda"),
    }
    ws, nbytes = layer.workspace(T, moe.MODE_ROUTE)
    moe.moe_route_from_logits(layer.handle, Ld.data_ptr() if T else 0, T, {n: t.data_ptr() for n, t in bufs.items()},
                              ws, nbytes, layer.stream)
    torch.cuda.synchronize()
    out = {n: t.cpu().numpy() for n, t in bufs.items()}
    out["sorted_token"] = out["sorted_token"][: T * k]
    return out


def assert_routing_equal(got: dict, ref: dict):
    assert np.array_equal(got["topk_ids"], ref["ids"]), "top-k ids differ"
    assert np.array_equal(got["topk_w"].view(np.uint32), ref["w"].view(np.uint32)), "gate weights differ"
    assert np.array_equal(got["expert_offsets"], ref["offsets"]), "expert offsets differ"
    assert np.array_equal(got["sorted_token"], ref["sorted_token"]), "sorted_token differs"
    assert np.array_equal(got["inv_row"], ref["inv_row"]), "inv_row differs"


def count_routing_switches(gpu_ids: np.ndarray, L_oracle: np.ndarray, k: int) -> int:
    """Route the oracle on its own fp32 logits (an independent run, not the
    GPU's logits) and compare the ordered top-k with the GPU's.  Every token
    whose routing differs must be a near-tie: at the first rank where the two
    lists part, the oracle's logit of its expert exceeds that of the GPU's
    by at most the sum of the two logits' tolerances, 2e-5 * (1 + |L|)
    (both sides are within 1e-5 * (1 + |L|) of the exact logit, which the
    tests assert separately).  Returns the number of such tokens."""
    import oracle
    ref = oracle.route_from_logits(L_oracle, k)["ids"]
    diff = np.nonzero((ref != gpu_ids).any(axis=1))[0]
    for t in diff:
        p = int(np.nonzero(ref[t] != gpu_ids[t])[0][0])
        a, b = int(ref[t, p]), int(gpu_ids[t, p])
        la, lb = float(L_oracle[t, a]), float(L_oracle[t, b])
        assert 0.0 <= la - lb <= 2e-5 * (1.0 + max(abs(la), abs(lb))), (int(t), p, a, b, la, lb)
    print(f"[routing] tokens routed differently under the oracle's own logits: {len(diff)} of {len(ref)}")
    return len(diff)


REL_L2_TOL = 5e-3          # relative L2 error of y
MAX_ABS_TOL = 3e-2         # max abs error / rms(y_oracle)


def compare_y(y_gpu: np.ndarray, y_ref: np.ndarray):
    """Tolerance of the layer output (bf16): rel-L2 <= 5e-3 and max abs
    error <= 3e-2 * rms(y_ref).  Returns (rel_l2, max_abs/rms)."""
    a = synth.bf16_to_f32(y_gpu).astype(np.float64)
    b = synth.bf16_to_f32(y_ref).astype(np.float64)
    assert np.all(np.isfinite(a)), "non-finite output"
    rms = np.sqrt(np.mean(b * b))
    rel = np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30)
    mx = np.max(np.abs(a - b)) / max(rms, 1e-30) if a.size else 0.0
    print(f"[parity] rel_l2={rel:.3e} max_abs/rms={mx:.3e} n={a.size}")
    assert rel <= REL_L2_TOL, f"relative L2 error {rel:.3e} > {REL_L2_TOL}"
    assert mx <= MAX_ABS_TOL, f"max abs error {mx:.3e} * rms > {MAX_ABS_TOL}"
    return rel, mx


def oracle_y(inp: dict, k: int, ids, w, rows=None):
    return oracle.forward(inp, k, ids, w, rows=rows)


def _e4m3_neighbours(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """True where codes a and b are adjacent values of the E4M3FN grid."""
    va, vb = oracle.e4m3_decode(a), oracle.e4m3_decode(b)
    lo, hi = np.minimum(va, vb), np.maximum(va, vb)
    grid = np.unique(oracle.e4m3_decode(np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)))
    return np.searchsorted(grid, hi) - np.searchsorted(grid, lo) == 1


H_BAND = 1e-5       # band around an E4M3 rounding midpoint, as a fraction of the block amax
SCALE_REL = 4e-6    # relative agreement of the h scales (amax / 448)


def check_h_codes(gpu_hq, gpu_sh, ref: dict, max_frac: float = 1e-3):
    """The GPU's h codes must equal the oracle's, except where the oracle's
    h sits within H_BAND (of its 128-block's amax) of the rounding midpoint
    between two adjacent E4M3 values: there the summation order decides and
    either code is correct.  Scales (amax/448 per 128 values) within
    SCALE_REL; at most max_frac of the codes may differ."""
    h32, hq, sh = ref["h32"], ref["hq"], ref["sh"]
    assert gpu_hq.shape == hq.shape and gpu_sh.shape == sh.shape
    srel = np.abs(gpu_sh.astype(np.float64) - sh) / np.abs(sh)
    # codes that differ but decode to the same value are -0 and +0: h/s rounded
    # to zero from either side of it, the same contribution to y
    diff = gpu_hq != hq
    signed_zero = diff & ((gpu_hq & 0x7F) == 0) & ((hq & 0x7F) == 0)
    diff &= ~signed_zero
    n = int(diff.sum())
    dist = np.zeros(0)
    if n:
        ratio = (h32.astype(np.float64) / np.repeat(sh.astype(np.float64), 128, axis=-1))[diff]
        va, vb = oracle.e4m3_decode(gpu_hq[diff]), oracle.e4m3_decode(hq[diff])
        mid, step = 0.5 * (va + vb), np.abs(va - vb)
        dist = np.abs(ratio - mid) / np.maximum(step, 1e-30)
        hmag = np.abs(ratio) / 448.0
    print(f"[h-codes] flips={n}/{hq.size} (+-0: {int(signed_zero.sum())}) max_scale_rel={srel.max():.2e} "
          f"max_dist/step={dist.max() if n else 0:.2e} "
          f"flip |h|/amax: {np.array2string(hmag[:8], precision=3) if n else '-'}")
    # The GPU forms h in fp32 from fp32 sums of 128-block partials, so its h
    # carries an absolute error of order 1e-6 of the block's amax (the
    # largest terms it sums); the oracle's h is fp64 rounded once.  A code
    # may therefore differ only where the oracle's scaled value h/s (range
    # +-448) lies within 448 * H_BAND of the midpoint between the two
    # codes, and the 1x128 scales (amax/448) agree to SCALE_REL.
    assert np.all(srel <= SCALE_REL), "h scales differ beyond rounding"
    if n:
        assert np.all(_e4m3_neighbours(gpu_hq[diff], hq[diff])), "an h code differs by more than one step"
        assert np.all(np.abs(ratio - mid) <= 448.0 * H_BAND), "an h code differs away from a rounding boundary"
    assert n <= max_frac * hq.size, f"{n} boundary flips out of {hq.size}"
    return n


def check_layer_output(inp: dict, k: int, dbg: dict, y_gpu: np.ndarray, rows=None):
    """Layer parity on the tokens `rows` (all when None), with the oracle
    routed by the GPU's logits (dbg ids/w were checked against the oracle's
    routing by the caller).

    1) Against the oracle with its own h: rel-L2 <= 5e-3 against its bf16
       y; on the tokens whose h codes all equal the GPU's, max-abs <=
       3e-2 * rms against its unrounded fp64 y (the bf16 rounding of y costs
       at most half a bf16 step).  The max-abs over all tokens is printed:
       one boundary-flipped code of a large h moves its token's y by up to
       a few 1e-2 * rms, so that figure is not bounded by 3e-2.
    2) Its h codes against the GPU's: equal except at rounding boundaries
       (check_h_codes).
    3) Against the oracle evaluated with the GPU's h codes (the other valid
       result at those boundaries): rel-L2 <= 5e-3 and max-abs <= 3e-2 * rms,
       both against bf16 y.  Only tokens with a flipped code need the second
       evaluation; for the others it equals the first bit for bit.
    Returns (rel_l2, max_abs/rms) of 3)."""
    ids, w = dbg["topk_ids"], dbg["topk_w"]
    y_ref, y64, href = oracle.forward(inp, k, ids, w, rows=rows, want_f64=True, want_h=True)
    sel = np.arange(y_gpu.shape[0]) if rows is None else np.asarray(rows)
    a = synth.bf16_to_f32(y_gpu[sel]).astype(np.float64)
    b = synth.bf16_to_f32(y_ref).astype(np.float64)
    rms = np.sqrt(np.mean(y64 * y64))
    rel_plain = np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30)
    err = np.abs(a - y64).max(axis=1) / max(rms, 1e-30) if a.size else np.zeros(sel.size)
    flips = check_h_codes(dbg["hq"][sel], dbg["sh"][sel], href)
    changed = np.nonzero((dbg["hq"][sel] != href["hq"]).reshape(sel.size, -1).any(axis=1))[0]
    same = np.ones(sel.size, bool)
    same[changed] = False
    mx_same = float(err[same].max()) if same.any() else 0.0
    print(f"[parity] own-h rel_l2={rel_plain:.3e} max_abs(vs fp64)/rms={float(err.max()) if err.size else 0:.3e} "
          f"(tokens without h flips: {mx_same:.3e}) h boundary flips={flips} tokens={sel.size} "
          f"tokens with a flip={changed.size}")
    assert rel_plain <= REL_L2_TOL, f"relative L2 error {rel_plain:.3e} > {REL_L2_TOL} (oracle's own h)"
    assert mx_same <= MAX_ABS_TOL, f"max abs error {mx_same:.3e} * rms > {MAX_ABS_TOL} (oracle's own h, fp64 y)"
    y_ov = y_ref.copy()
    if changed.size:
        y_ov[changed] = oracle.forward(inp, k, ids, w, rows=sel[changed], hq_in=dbg["hq"], sh_in=dbg["sh"])
    return compare_y(y_gpu[sel], y_ov)


def single_expert_inputs(inp: dict) -> dict:
    """The layer's inputs without the shared expert: with k = 1 and a given
    (expert, weight) per token, the oracle then computes that one expert's
    weighted output for each token."""
    return {n: v for n, v in inp.items() if not n.startswith("sh_")}


def check_hot_expert(layer, inp: dict, k: int, dbg: dict, x_bits: np.ndarray, mode: int, expert: int):
    """Every token routed to `expert`, checked on that expert alone: the
    layer runs with the slot of `expert` deferred (moe_forward_deferred, same
    GEMMs, split combine), so y_next[t] = bf16(w O_expert(t)); the oracle
    evaluates only that expert for each such token (k = 1, no shared
    expert).  Against the oracle's own h: rel-L2 <= 5e-3.  Against the
    oracle's unrounded fp64 value under the GPU's h codes (its own h where
    the codes agree): every element within half a bf16 step of it plus
    3e-3 * rms -- the bf16 rounding of the output plus the error of the
    tensor core's FP8 partial sums, which is absolute (of the order of the
    summed terms, not of a result that cancels to near zero).  (The
    layer's 3e-2 * rms max-abs bound alone is not the right scale here: one
    expert's weighted output has heavier tails than the layer output, and
    a rounding tie decided the other way at an element of many times the
    rms is a full bf16 step.)"""
    T, H = x_bits.shape
    ids, w = dbg["topk_ids"], dbg["topk_w"]
    mask = (ids == expert).astype(np.uint8)
    toks = np.nonzero(mask.any(axis=1))[0].astype(np.int32)
    slot = np.argmax(mask[toks], axis=1)
    x = to_dev(x_bits.view(np.int16))
    y_now, y_next = torch.empty_like(x), torch.empty_like(x)
    m = to_dev(mask)
    ws, nb = layer.workspace(T, mode)
    moe.moe_forward_deferred(layer.handle, mode, x.data_ptr(), T, m.data_ptr(), y_now.data_ptr(), y_next.data_ptr(),
                             ws, nb, layer.stream)
    torch.cuda.synchronize()
    st, flags = moe.moe_get_device_status(layer.handle, layer.stream)
    assert st == 0 and flags == 0, f"device status {st} flags {flags:#x}"
    y_gpu = y_next.cpu().numpy().view(np.uint16)[toks]
    del y_now, y_next, x, m
    one = single_expert_inputs(inp)
    ids1 = np.zeros((T, 1), np.int32)
    w1 = np.zeros((T, 1), np.float32)
    ids1[toks, 0] = expert
    w1[toks, 0] = w[toks, slot]
    y_ref, y64, href = oracle.forward(one, 1, ids1, w1, rows=toks, want_f64=True, want_h=True)
    a = synth.bf16_to_f32(y_gpu).astype(np.float64)
    b = synth.bf16_to_f32(y_ref).astype(np.float64)
    rel_plain = np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30)
    ghq = dbg["hq"][toks, slot][:, None, :]
    gsh = dbg["sh"][toks, slot][:, None, :]
    flips = check_h_codes(ghq, gsh, href)
    changed = np.nonzero((ghq != href["hq"]).reshape(toks.size, -1).any(axis=1))[0]
    y64_ov = y64.copy()
    if changed.size:
        hq_full = np.zeros((T, 1, ghq.shape[-1]), np.uint8)
        sh_full = np.ones((T, 1, gsh.shape[-1]), np.float32)
        hq_full[toks] = ghq
        sh_full[toks] = gsh
        _, y64_ov[changed] = oracle.forward(one, 1, ids1, w1, rows=toks[changed], hq_in=hq_full, sh_in=sh_full,
                                            want_f64=True)
    rms = np.sqrt(np.mean(y64_ov * y64_ov))
    mag = np.abs(y64_ov)
    half_step = np.ldexp(1.0, np.floor(np.log2(np.maximum(mag, 1e-300))).astype(np.int64) - 8)
    err = np.abs(a - y64_ov)
    worst = float(np.max(err / (half_step + 3e-3 * rms)))
    rel_ov = np.linalg.norm(a - y64_ov) / max(np.linalg.norm(y64_ov), 1e-30)
    print(f"[hot expert {expert}] tokens={toks.size} own-h rel_l2={rel_plain:.3e} h flips={flips} "
          f"vs fp64 (GPU h): rel_l2={rel_ov:.3e} max_abs/rms={float(err.max()) / rms:.3e} "
          f"max err / (half bf16 step + 3e-3 rms)={worst:.3f}")
    assert rel_plain <= REL_L2_TOL and rel_ov <= REL_L2_TOL
    assert worst <= 1.0, "an element is further than half a bf16 step from the oracle's fp64 value"
    return toks.size
