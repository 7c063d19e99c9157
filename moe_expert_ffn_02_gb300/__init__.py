"""Python binding of libmoe.so, the GB300 (sm_103a) routed-expert MoE FFN layer.

Argument marshalling only: every step of the layer runs in the library's
CUDA kernels.  The functions carry the C ABI's names (include/moe.h) and take
plain integers for device pointers and streams, so any allocator can feed
them; the `Layer` helper adds torch-tensor convenience on top (torch is used
for device memory and streams, nothing else).

There is no fallback: if libmoe.so is missing or cannot be loaded, every
call raises MoeError.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

__all__ = [
    "MoeError", "MoeDesc", "MoeWeights", "MoeRouteOut", "MODE_ROUTE", "MODE_PREFILL", "MODE_DECODE",
    "DECODE_MAX_T", "moe_create", "moe_destroy", "moe_workspace_bytes", "moe_route", "moe_route_from_logits",
    "moe_route_from_logits_noalloc", "moe_forward_prefill", "moe_forward_decode", "moe_forward_host", "moe_get_device_status",
    "moe_set_wait_limit", "moe_debug_timeout_probe", "moe_debug_inject", "moe_profile_enable", "moe_profile_read", "moe_status_string", "moe_last_error",
    "moe_abi_version", "moe_forward_smallep", "moe_forward_deferred", "moe_layers_workspace_bytes",
    "moe_forward_layers", "smallep_groups", "moe_create_ex", "moe_tiles_bytes", "moe_tiles_load", "moe_forward_tiles",
    "CREATE_HOST_TILES", "library_path", "load", "Layer", "LayerStackGraph", "StreamedStack",
]

MODE_ROUTE, MODE_PREFILL, MODE_DECODE = 0, 1, 2
CREATE_HOST_TILES = 1
DECODE_MAX_T = 64
MOE_OK = 0
DEV_BAD_EXPERT_ID, DEV_BAD_ROW, DEV_WAIT_TIMEOUT = 0x1, 0x2, 0x4


class MoeError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{message} (status {status})")
        self.status = status


class MoeDesc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("hidden", "inter", "n_experts", "top_k", "n_shared", "shared_inter")]


class MoeWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "router_w", "router_bias", "w_gate", "w_up", "w_down", "s_gate", "s_up", "s_down",
        "sh_gate", "sh_up", "sh_down", "sh_s_gate", "sh_s_up", "sh_s_down")]


class MoeRouteOut(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "logits", "topk_ids", "topk_w", "expert_offsets", "sorted_token", "inv_row", "xq", "sx", "hq", "sh")]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False):
    """Load libmoe.so (optionally building it first).  The environment
    variable MOE_LIBRARY, if set, names another build of the library to load."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = os.environ.get("MOE_LIBRARY") or _build.LIB
        if build_if_missing and path == _build.LIB and not _build.up_to_date():
            _build.build()
        if not os.path.exists(path):
            raise MoeError(-1, f"libmoe.so is not built ({path}); run __graft_entry__.build() first")
        try:
            lib = ctypes.CDLL(path)
        except OSError as e:
            raise MoeError(-1, f"cannot load {path}: {e}") from e
        vp, i32, u32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint32, ctypes.c_size_t
        st = ctypes.c_int
        sig = {
            "moe_create": ([ctypes.POINTER(MoeDesc), ctypes.POINTER(MoeWeights), vp, ctypes.POINTER(vp)], st),
            "moe_destroy": ([vp], st),
            "moe_workspace_bytes": ([vp, i32, i32, ctypes.POINTER(sz)], st),
            "moe_route": ([vp, vp, i32, ctypes.POINTER(MoeRouteOut), vp, sz, vp], st),
            "moe_route_from_logits": ([vp, vp, i32, ctypes.POINTER(MoeRouteOut), vp, sz, vp], st),
            "moe_forward_prefill": ([vp, vp, i32, vp, ctypes.POINTER(MoeRouteOut), vp, sz, vp], st),
            "moe_forward_decode": ([vp, vp, i32, vp, ctypes.POINTER(MoeRouteOut), vp, sz, vp], st),
            "moe_forward_host": ([vp, i32, vp, i32, vp, vp, sz, vp], st),
            "moe_get_device_status": ([vp, vp, ctypes.POINTER(u32)], st),
            "moe_set_wait_limit": ([vp, u32], st),
            "moe_debug_timeout_probe": ([vp, vp], st),
            "moe_debug_inject": ([vp, u32], st),
            "moe_route_from_logits_noalloc": ([vp, vp, i32, ctypes.POINTER(MoeRouteOut), vp], st),
            "moe_forward_smallep": ([vp, i32, i32, vp, i32, vp, vp, sz, vp], st),
            "moe_create_ex": ([ctypes.POINTER(MoeDesc), ctypes.POINTER(MoeWeights), u32, vp, ctypes.POINTER(vp)], st),
            "moe_tiles_bytes": ([vp, ctypes.POINTER(sz)], st),
            "moe_tiles_load": ([vp, vp, vp], st),
            "moe_forward_tiles": ([vp, i32, vp, vp, i32, vp, vp, sz, vp], st),
            "moe_forward_deferred": ([vp, i32, vp, i32, vp, vp, vp, vp, sz, vp], st),
            "moe_layers_workspace_bytes": ([ctypes.POINTER(vp), i32, i32, i32, ctypes.POINTER(sz)], st),
            "moe_forward_layers": ([ctypes.POINTER(vp), i32, i32, vp, i32, vp, vp, sz, vp], st),
            "moe_profile_enable": ([vp, i32], st),
            "moe_profile_read": ([vp, ctypes.POINTER(ctypes.c_float), i32], st),
            "moe_status_string": ([st], ctypes.c_char_p),
            "moe_last_error": ([], ctypes.c_char_p),
            "moe_abi_version": ([], i32),
        }
        for name, (args, res) in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def _check(status: int):
    if status != MOE_OK:
        lib = load()
        raise MoeError(status, f"{lib.moe_status_string(status).decode()}: {lib.moe_last_error().decode()}")


def _route_out(out):
    if out is None:
        return None
    if isinstance(out, MoeRouteOut):
        return ctypes.byref(out)
    return ctypes.byref(MoeRouteOut(**{k: v for k, v in out.items() if v}))


# ---------------------------------------------------------------- ABI functions

def moe_abi_version() -> int:
    return int(load().moe_abi_version())


def moe_status_string(status: int) -> str:
    return load().moe_status_string(status).decode()


def moe_last_error() -> str:
    return load().moe_last_error().decode()


def moe_create(desc: MoeDesc, weights: MoeWeights, stream: int = 0) -> int:
    h = ctypes.c_void_p()
    _check(load().moe_create(ctypes.byref(desc), ctypes.byref(weights), stream, ctypes.byref(h)))
    return h.value


def moe_create_ex(desc: MoeDesc, weights: MoeWeights, flags: int, stream: int = 0) -> int:
    h = ctypes.c_void_p()
    _check(load().moe_create_ex(ctypes.byref(desc), ctypes.byref(weights), flags, stream, ctypes.byref(h)))
    return h.value


def moe_tiles_bytes(layer: int) -> int:
    n = ctypes.c_size_t()
    _check(load().moe_tiles_bytes(layer, ctypes.byref(n)))
    return n.value


def moe_tiles_load(layer: int, slot: int, stream: int = 0) -> None:
    _check(load().moe_tiles_load(layer, slot, stream))


def moe_forward_tiles(layer: int, mode: int, slot: int, x: int, T: int, y: int, ws: int, ws_bytes: int,
                      stream: int = 0) -> None:
    _check(load().moe_forward_tiles(layer, mode, slot, x, T, y, ws, ws_bytes, stream))


def moe_destroy(layer: int) -> None:
    _check(load().moe_destroy(layer))


def moe_workspace_bytes(layer: int, T: int, mode: int) -> int:
    n = ctypes.c_size_t()
    _check(load().moe_workspace_bytes(layer, T, mode, ctypes.byref(n)))
    return n.value


def moe_route(layer: int, x: int, T: int, out, ws: int, ws_bytes: int, stream: int = 0) -> None:
    _check(load().moe_route(layer, x, T, _route_out(out), ws, ws_bytes, stream))


def moe_route_from_logits(layer: int, logits: int, T: int, out, ws: int, ws_bytes: int, stream: int = 0) -> None:
    _check(load().moe_route_from_logits(layer, logits, T, _route_out(out), ws, ws_bytes, stream))


def moe_route_from_logits_noalloc(layer: int, logits: int, T: int, out, stream: int = 0) -> None:
    """Routing from given logits with the library's built-in scratch (no
    workspace, no allocation) -- for callers that cannot allocate device
    memory when they route.  See include/moe.h for the size limit."""
    _check(load().moe_route_from_logits_noalloc(layer, logits, T, _route_out(out), stream))


def moe_forward_prefill(layer: int, x: int, T: int, y: int, dbg, ws: int, ws_bytes: int, stream: int = 0) -> None:
    _check(load().moe_forward_prefill(layer, x, T, y, _route_out(dbg), ws, ws_bytes, stream))


def moe_forward_decode(layer: int, x: int, T: int, y: int, dbg, ws: int, ws_bytes: int, stream: int = 0) -> None:
    _check(load().moe_forward_decode(layer, x, T, y, _route_out(dbg), ws, ws_bytes, stream))


def moe_forward_host(layer: int, mode: int, x_host: int, T: int, y_host: int, ws: int, ws_bytes: int,
                     stream: int = 0) -> None:
    _check(load().moe_forward_host(layer, mode, x_host, T, y_host, ws, ws_bytes, stream))


def moe_forward_smallep(layer: int, mode: int, n_ranks: int, x: int, T: int, y: int, ws: int, ws_bytes: int,
                        stream: int = 0) -> None:
    _check(load().moe_forward_smallep(layer, mode, n_ranks, x, T, y, ws, ws_bytes, stream))


def smallep_groups(n_experts: int, n_ranks: int):
    """Expert range [lo, hi) of each SmallEP rank, as moe_forward_smallep
    splits them: rank p holds [ceil(p E / P), ceil((p + 1) E / P)); rank 0
    also holds the shared expert."""
    b = [(p * n_experts + n_ranks - 1) // n_ranks for p in range(n_ranks + 1)]
    return [(b[p], b[p + 1]) for p in range(n_ranks)]


def moe_forward_deferred(layer: int, mode: int, x: int, T: int, defer: int, y_now: int, y_next: int, ws: int,
                         ws_bytes: int, stream: int = 0) -> None:
    _check(load().moe_forward_deferred(layer, mode, x, T, defer, y_now, y_next, ws, ws_bytes, stream))


def _handles(layers):
    arr = (ctypes.c_void_p * len(layers))(*[int(h) for h in layers])
    return arr


def moe_layers_workspace_bytes(layers, T: int, mode: int) -> int:
    n = ctypes.c_size_t()
    _check(load().moe_layers_workspace_bytes(_handles(layers), len(layers), T, mode, ctypes.byref(n)))
    return n.value


def moe_forward_layers(layers, mode: int, x: int, T: int, y: int, ws: int, ws_bytes: int, stream: int = 0) -> None:
    _check(load().moe_forward_layers(_handles(layers), len(layers), mode, x, T, y, ws, ws_bytes, stream))


def moe_get_device_status(layer: int, stream: int = 0):
    """Returns (status, flags) without raising, so callers can inspect both."""
    f = ctypes.c_uint32()
    st = load().moe_get_device_status(layer, stream, ctypes.byref(f))
    return int(st), int(f.value)


def moe_set_wait_limit(layer: int, microseconds: int) -> None:
    _check(load().moe_set_wait_limit(layer, microseconds))


def moe_debug_timeout_probe(layer: int, stream: int = 0) -> None:
    _check(load().moe_debug_timeout_probe(layer, stream))


def moe_debug_inject(layer: int, faults: int) -> None:
    """Plant the faults (DEV_BAD_EXPERT_ID | DEV_BAD_ROW) in the next routing
    or forward call's workspace; the kernels must flag them and stay in
    bounds (test hook, see include/moe.h)."""
    _check(load().moe_debug_inject(layer, faults))


PROFILE_STAGES = ("route", "quant_x", "gate_up", "down", "combine")


PROFILE_SELECT = 0x40000000


def moe_profile_enable(layer: int, enable: bool = True, stages=None) -> None:
    """Record stage events in forward calls: every stage, or only the named
    ones (e.g. stages=("gate_up",)); enable=False turns profiling off."""
    if not enable:
        code = 0
    elif stages is None:
        code = 1
    else:
        code = PROFILE_SELECT
        for name in stages:
            code |= 1 << PROFILE_STAGES.index(name)
    _check(load().moe_profile_enable(layer, code))


def moe_profile_read(layer: int):
    """Elapsed ms of each stage of the most recent forward call (dict); -1
    for a stage that is not timed."""
    buf = (ctypes.c_float * len(PROFILE_STAGES))()
    _check(load().moe_profile_read(layer, buf, len(PROFILE_STAGES)))
    return dict(zip(PROFILE_STAGES, [float(v) for v in buf]))


# ---------------------------------------------------------------- torch convenience

class Layer:
    """A layer built from torch CUDA tensors (checkpoint layout, see moe.h).

    weights: dict with router_w, router_b (or None), w_gate, w_up, w_down,
    s_gate, s_up, s_down and, with a shared expert, sh_* of the same layout.
    The library copies the weights; the tensors may be freed afterwards.
    """

    def __init__(self, hidden, inter, n_experts, top_k, weights: dict, n_shared: int = 1, stream=None,
                 host_tiles: bool = False):
        import torch
        self.desc = MoeDesc(hidden, inter, n_experts, top_k, n_shared, inter if n_shared else 0)
        p = lambda n: (weights[n].data_ptr() if weights.get(n) is not None else None)
        self.weights = MoeWeights(
            p("router_w"), p("router_b"), p("w_gate"), p("w_up"), p("w_down"), p("s_gate"), p("s_up"), p("s_down"),
            p("sh_gate"), p("sh_up"), p("sh_down"), p("sh_s_gate"), p("sh_s_up"), p("sh_s_down"))
        self.stream = stream if stream is not None else torch.cuda.current_stream().cuda_stream
        self.handle = moe_create_ex(self.desc, self.weights, CREATE_HOST_TILES if host_tiles else 0, self.stream)
        self._ws = {}

    def workspace(self, T: int, mode: int):
        import torch
        need = moe_workspace_bytes(self.handle, T, mode)
        if mode == MODE_PREFILL or mode == MODE_DECODE:
            need += 4 * T * self.desc.hidden + 1024     # room for moe_forward_host's device copies
        cur = self._ws.get("buf")
        if cur is None or cur.numel() < need:
            self._ws["buf"] = torch.empty(max(need, 256), dtype=torch.uint8, device="cuda")
        buf = self._ws["buf"]
        return buf.data_ptr(), buf.numel()

    def close(self):
        if self.handle:
            moe_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class LayerStackGraph:
    """A stack of layers (handles) run as one moe_forward_layers call,
    captured once into a CUDA graph and replayed: the whole decode step is a
    single graph launch.  x and y are torch CUDA bf16-bits tensors [T][H]
    owned by the caller; replay() runs the stack on the current contents of
    x and leaves the result in y."""

    def __init__(self, handles, mode: int, x, y, warmup: int = 1):
        import torch
        self.handles = list(handles)
        self.mode = mode
        self.x, self.y = x, y
        T = x.shape[0]
        need = moe_layers_workspace_bytes(self.handles, T, mode)
        self.ws = torch.empty(max(need, 256), dtype=torch.uint8, device=x.device)
        self.stream = torch.cuda.Stream(device=x.device)
        run = lambda: moe_forward_layers(self.handles, mode, x.data_ptr(), T, y.data_ptr(), self.ws.data_ptr(),
                                         self.ws.numel(), self.stream.cuda_stream)
        with torch.cuda.stream(self.stream):
            for _ in range(warmup):           # one-time kernel attributes are set outside the capture
                run()
        self.stream.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=self.stream):
            run()

    def replay(self):
        """Launch the captured stack on the current torch stream."""
        self.graph.replay()


class StreamedStack:
    """A stack of host-tile layers (moe_create_ex with CREATE_HOST_TILES) run
    through a two-slot device ring: while layer l computes from slot l % 2,
    a copy stream loads layer l + 1's tiles into the other slot (ordered by
    events: a slot is reloaded only after the layer that read it finished).
    x and y: torch CUDA [T][H] bf16-bits tensors; run() computes on the
    current torch stream and returns when the work is enqueued."""

    def __init__(self, layers, mode: int, x, y):
        import torch
        self.layers = list(layers)
        self.mode, self.x, self.y = mode, x, y
        T = x.shape[0]
        slot_bytes = max(moe_tiles_bytes(ly.handle) for ly in self.layers)
        self.slots = [torch.empty(slot_bytes, dtype=torch.uint8, device=x.device) for _ in range(2)]
        self.acts = [torch.empty_like(x) for _ in range(2)]
        need = max(moe_workspace_bytes(ly.handle, T, mode) for ly in self.layers)
        self.ws = torch.empty(max(need, 256), dtype=torch.uint8, device=x.device)
        self.copy = torch.cuda.Stream(device=x.device)
        self.loaded = [torch.cuda.Event() for _ in range(2)]
        self.done = [torch.cuda.Event() for _ in range(2)]

    def run(self):
        import torch
        comp = torch.cuda.current_stream()
        n, T = len(self.layers), self.x.shape[0]

        def load_into(l):
            s = l % 2
            self.copy.wait_event(self.done[s]) if l >= 2 else self.copy.wait_stream(comp)
            moe_tiles_load(self.layers[l].handle, self.slots[s].data_ptr(), self.copy.cuda_stream)
            self.loaded[s].record(self.copy)

        load_into(0)
        for l in range(n):
            if l + 1 < n:
                load_into(l + 1)
            s = l % 2
            comp.wait_event(self.loaded[s])
            src = self.x if l == 0 else self.acts[(l - 1) % 2]
            dst = self.y if l == n - 1 else self.acts[l % 2]
            moe_forward_tiles(self.layers[l].handle, self.mode, self.slots[s].data_ptr(), src.data_ptr(), T,
                              dst.data_ptr(), self.ws.data_ptr(), self.ws.numel(), comp.cuda_stream)
            self.done[s].record(comp)
