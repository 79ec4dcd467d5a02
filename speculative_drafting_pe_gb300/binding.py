"""Thin ctypes binding of libpe.so (C ABI in include/pe.h).

Argument marshalling only: every step of the draft pass and of the
verify/rebuild runs in the library's CUDA kernels. PyTorch supplies device
memory and the current stream. ``load()`` raises if the library is missing;
there is no fallback path.
"""

import ctypes
import os

import torch

from . import build as _build

PE_OK = 0
PE_REQ_OK, PE_REQ_CAPACITY, PE_REQ_BAD_PAGE, PE_REQ_BAD_INPUT = 0, 1, 2, 3
PE_DTYPE_BF16, PE_DTYPE_FP32, PE_DTYPE_FP8W = 0, 1, 2
PE_DEVERR_GEMM_TIMEOUT, PE_DEVERR_ATTN_TIMEOUT, PE_DEVERR_CHAIN_TIMEOUT = 1, 2, 4
PE_DRAFT_PARALLEL, PE_DRAFT_SEQUENTIAL = 0, 1

EXPORTS = (
    "pe_init_drafter", "pe_draft", "pe_verify_rebuild", "pe_device_errors",
    "pe_last_launch_count", "pe_destroy", "pe_last_error", "pe_abi_version", "pe_linear_scratch", "pe_linear",
    "pe_profile_start", "pe_profile_stop", "pe_kernel_name",
    "pe_step_graph_create", "pe_step_graph_launch", "pe_step_graph_launch_count", "pe_step_graph_destroy",
    "pe_linear_noalloc", "pe_test_stall_chain", "pe_draft_sequential", "pe_step_graph_create_ex",
    "pe_init_drafter_fp8", "pe_linear_fp8", "pe_draft_refeed", "pe_verify_rebuild_refeed",
    "pe_sample_drafts", "pe_verify_stochastic",
)
KERNEL_KINDS = ("fc", "row_build", "rmsnorm", "qkv", "attention", "o_proj", "gate_up", "down", "lm_head", "argmax",
                "layer_chain")

_i32 = ctypes.c_int32
_vp = ctypes.c_void_p


class PeConfig(ctypes.Structure):
    _fields_ = [("hidden", _i32), ("n_layers", _i32), ("n_q_heads", _i32), ("n_kv_heads", _i32),
                ("head_dim", _i32), ("ffn", _i32), ("vocab", _i32), ("rms_eps", ctypes.c_float),
                ("rope_theta", ctypes.c_float), ("page_size", _i32), ("k_max", _i32), ("dtype", _i32)]


_LAYER_FIELDS = ("norm_e", "norm_h", "attn_norm", "w_qkv", "w_o", "mlp_norm", "w_gate", "w_up", "w_down")


class PeLayerWeights(ctypes.Structure):
    _fields_ = [(n, _vp) for n in _LAYER_FIELDS]


_TOP_FIELDS = ("fc", "embed", "emb_mask", "h_shared", "final_norm", "lm_head")


class PeWeights(ctypes.Structure):
    _fields_ = [(n, _vp) for n in _TOP_FIELDS] + [("layer", PeLayerWeights * 4)]


_LAYER_SCALE_FIELDS = ("w_qkv", "w_o", "w_gate", "w_up", "w_down")


class PeLayerScales(ctypes.Structure):
    _fields_ = [(n, _vp) for n in _LAYER_SCALE_FIELDS]


class PeWeightScales(ctypes.Structure):
    _fields_ = [("fc", _vp), ("lm_head", _vp), ("layer", PeLayerScales * 4)]


class PeError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"libpe error {code}: {msg}")
        self.code = code


_LIB = None


def library_path():
    return _build.LIB


def load():
    """Load libpe.so (built by ``__graft_entry__.build()``); raise if absent."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"libpe.so not found at {path}; build it with __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    lib.pe_abi_version.restype = ctypes.c_int
    lib.pe_last_error.restype = ctypes.c_char_p
    lib.pe_init_drafter.argtypes = [ctypes.POINTER(PeConfig), ctypes.POINTER(PeWeights), _i32, _i32,
                                    ctypes.POINTER(_vp)]
    lib.pe_init_drafter.restype = ctypes.c_int
    lib.pe_init_drafter_fp8.argtypes = [ctypes.POINTER(PeConfig), ctypes.POINTER(PeWeights),
                                        ctypes.POINTER(PeWeightScales), _i32, _i32, ctypes.POINTER(_vp)]
    lib.pe_init_drafter_fp8.restype = ctypes.c_int
    lib.pe_linear_fp8.argtypes = [_i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp]
    lib.pe_linear_fp8.restype = ctypes.c_int
    lib.pe_draft.argtypes = [_vp, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp]
    lib.pe_draft.restype = ctypes.c_int
    lib.pe_draft_refeed.argtypes = [_vp, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _vp, _vp,
                                    _vp, _vp, _vp, _vp]
    lib.pe_draft_refeed.restype = ctypes.c_int
    lib.pe_verify_rebuild_refeed.argtypes = [_vp, _i32, _i32, _vp, _vp, _vp, _i32, _i32, _vp, _vp, _vp, _vp, _vp,
                                             _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]
    lib.pe_verify_rebuild_refeed.restype = ctypes.c_int
    lib.pe_sample_drafts.argtypes = [_vp, _i32, _i32, _vp, ctypes.c_float, _vp, _vp, _vp, _vp]
    lib.pe_sample_drafts.restype = ctypes.c_int
    lib.pe_verify_stochastic.argtypes = [_vp, _i32, _i32, _vp, _vp, _vp, ctypes.c_float, _vp, _vp, _vp, _i32, _i32,
                                         _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]
    lib.pe_verify_stochastic.restype = ctypes.c_int
    lib.pe_draft_sequential.argtypes = lib.pe_draft.argtypes
    lib.pe_draft_sequential.restype = ctypes.c_int
    lib.pe_verify_rebuild.argtypes = [_vp, _i32, _i32, _vp, _vp, _vp, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp,
                                      _vp, _vp, _vp, _vp, _vp]
    lib.pe_verify_rebuild.restype = ctypes.c_int
    lib.pe_device_errors.argtypes = [_vp, _vp, ctypes.POINTER(ctypes.c_uint32)]
    lib.pe_device_errors.restype = ctypes.c_int
    lib.pe_last_launch_count.argtypes = [_vp]
    lib.pe_last_launch_count.restype = ctypes.c_int
    lib.pe_destroy.argtypes = [_vp]
    lib.pe_destroy.restype = None
    lib.pe_linear_scratch.argtypes = [_i32, _i32, _i32, _i32, ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(_i32)]
    lib.pe_linear_scratch.restype = ctypes.c_int
    lib.pe_linear.argtypes = [_i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp]
    lib.pe_linear.restype = ctypes.c_int
    lib.pe_linear_noalloc.argtypes = [_i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp]
    lib.pe_linear_noalloc.restype = ctypes.c_int
    lib.pe_test_stall_chain.argtypes = [_vp, _vp]
    lib.pe_test_stall_chain.restype = ctypes.c_int
    lib.pe_profile_start.argtypes = [_vp, _i32, _i32]
    lib.pe_profile_start.restype = ctypes.c_int
    lib.pe_profile_stop.argtypes = [_vp, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(_i32)]
    lib.pe_profile_stop.restype = ctypes.c_int
    lib.pe_kernel_name.argtypes = [_i32]
    lib.pe_kernel_name.restype = ctypes.c_char_p
    lib.pe_step_graph_create.argtypes = [_vp, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _vp, _vp, _vp, _vp,
                                         _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.POINTER(_vp)]
    lib.pe_step_graph_create.restype = ctypes.c_int
    lib.pe_step_graph_create_ex.argtypes = [_vp, _i32] + lib.pe_step_graph_create.argtypes[1:]
    lib.pe_step_graph_create_ex.restype = ctypes.c_int
    lib.pe_step_graph_launch.argtypes = [_vp, _vp]
    lib.pe_step_graph_launch.restype = ctypes.c_int
    lib.pe_step_graph_launch_count.argtypes = [_vp]
    lib.pe_step_graph_launch_count.restype = ctypes.c_int
    lib.pe_step_graph_destroy.argtypes = [_vp]
    lib.pe_step_graph_destroy.restype = None
    _LIB = lib
    return lib


def _check(rc):
    if rc != PE_OK:
        raise PeError(rc, _LIB.pe_last_error().decode())


def _p(t):
    return None if t is None else _vp(t.data_ptr())


def _stream_ptr(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return _vp(s.cuda_stream)


def _need(t, dtype, device, name):
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if t.device != device:
        raise ValueError(f"{name}: expected device {device}, got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")


class Drafter:
    """A drafter handle over caller-owned device weights.

    shape: object with hidden, n_q_heads, n_kv_heads, head_dim, ffn, vocab,
    rms_eps, rope_theta, page_size, dtype ("bf16" | "fp32").
    weights: dict as produced by ``synth.make_weights`` with tensors on the
    device; the Drafter keeps references so they outlive the handle.
    """

    def __init__(self, shape, weights, max_batch, k_max, device=None, fp8_scales=None):
        """fp8_scales: per-row fp32 scales ({"fc", "lm_head", "layers": [...]})
        when the GEMM matrices of `weights` are E4M3 codes (uint8, as made by
        ``synth.quantize_weights_fp8``); the drafter then runs bf16 otherwise."""
        lib = load()
        self.shape = shape
        self.dtype = torch.bfloat16 if shape.dtype == "bf16" else torch.float32
        self.device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        self.k_max = k_max
        self.max_batch = max_batch
        self._weights = weights
        self._scales = fp8_scales
        fp8 = fp8_scales is not None
        if fp8 and self.dtype != torch.bfloat16:
            raise ValueError("FP8 weights go with a bf16 drafter shape")
        cfg = PeConfig(shape.hidden, 4, shape.n_q_heads, shape.n_kv_heads, shape.head_dim, shape.ffn,
                       shape.vocab, shape.rms_eps, shape.rope_theta, shape.page_size, k_max,
                       PE_DTYPE_FP8W if fp8 else (PE_DTYPE_BF16 if shape.dtype == "bf16" else PE_DTYPE_FP32))
        gemm = {"fc", "lm_head", "w_qkv", "w_o", "w_gate", "w_up", "w_down"}
        w = PeWeights()
        for n in _TOP_FIELDS:
            t = weights[n]
            _need(t, torch.uint8 if fp8 and n in gemm else self.dtype, self.device, n)
            setattr(w, n, t.data_ptr())
        for li, L in enumerate(weights["layers"]):
            for n in _LAYER_FIELDS:
                t = L.get(n)
                if t is not None:
                    _need(t, torch.uint8 if fp8 and n in gemm else self.dtype, self.device, f"layers[{li}].{n}")
                    setattr(w.layer[li], n, t.data_ptr())
        self._cfg, self._w = cfg, w
        h = _vp()
        if fp8:
            sc = PeWeightScales()
            for n in ("fc", "lm_head"):
                _need(fp8_scales[n], torch.float32, self.device, f"scales.{n}")
                setattr(sc, n, fp8_scales[n].data_ptr())
            for li, L in enumerate(fp8_scales["layers"]):
                for n in _LAYER_SCALE_FIELDS:
                    _need(L[n], torch.float32, self.device, f"scales.layers[{li}].{n}")
                    setattr(sc.layer[li], n, L[n].data_ptr())
            self._sc = sc
            _check(lib.pe_init_drafter_fp8(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(sc), max_batch,
                                           self.device.index or 0, ctypes.byref(h)))
        else:
            _check(lib.pe_init_drafter(ctypes.byref(cfg), ctypes.byref(w), max_batch, self.device.index or 0,
                                       ctypes.byref(h)))
        self._h = h

    def draft(self, last_token, target_hidden, positions, seq_lens, page_table, num_pages, k_cache, v_cache,
              K, drafts=None, status=None, logits=None, stream=None, sequential=False):
        """Enqueue one draft pass (K sequential one-row passes with
        sequential=True); returns (drafts [B, K] int32, status [B] int32)."""
        B = last_token.shape[0]
        dev = self.device
        for name, t in (("last_token", last_token), ("positions", positions), ("seq_lens", seq_lens),
                        ("page_table", page_table)):
            _need(t, torch.int32, dev, name)
        _need(target_hidden, self.dtype, dev, "target_hidden")
        _need(k_cache, self.dtype, dev, "k_cache")
        _need(v_cache, self.dtype, dev, "v_cache")
        if drafts is None:
            drafts = torch.empty(B, K, dtype=torch.int32, device=dev)
        if status is None:
            status = torch.empty(B, dtype=torch.int32, device=dev)
        if logits is not None:
            _need(logits, torch.float32, dev, "logits")
        fn = load().pe_draft_sequential if sequential else load().pe_draft
        _check(fn(self._h, B, K, _p(last_token), _p(target_hidden), _p(positions), _p(seq_lens),
                  _p(page_table), page_table.shape[1], num_pages, _p(k_cache), _p(v_cache),
                  _p(drafts), _p(logits), _p(status), _stream_ptr(stream)))
        return drafts, status

    def draft_refeed(self, tokens, n_real, target_hidden, positions, seq_lens, page_table, num_pages, k_cache,
                     v_cache, K, drafts=None, status=None, logits=None, stream=None):
        """Enqueue a draft pass with re-fed real rows: tokens [B, n_max]
        int32, n_real [B] int32, target_hidden [B, n_max, 3H]. Returns
        (drafts [B, K] int32, status [B] int32)."""
        B, n_max = tokens.shape
        dev = self.device
        for name, t in (("tokens", tokens), ("n_real", n_real), ("positions", positions), ("seq_lens", seq_lens),
                        ("page_table", page_table)):
            _need(t, torch.int32, dev, name)
        _need(target_hidden, self.dtype, dev, "target_hidden")
        if tuple(target_hidden.shape[:2]) != (B, n_max):
            raise ValueError("target_hidden must be [B, n_max, 3H]")
        if drafts is None:
            drafts = torch.empty(B, K, dtype=torch.int32, device=dev)
        if status is None:
            status = torch.empty(B, dtype=torch.int32, device=dev)
        if logits is not None:
            _need(logits, torch.float32, dev, "logits")
        _check(load().pe_draft_refeed(self._h, B, K, n_max, _p(tokens), _p(n_real), _p(target_hidden),
                                      _p(positions), _p(seq_lens), _p(page_table), page_table.shape[1], num_pages,
                                      _p(k_cache), _p(v_cache), _p(drafts), _p(logits), _p(status),
                                      _stream_ptr(stream)))
        return drafts, status

    def sample_drafts(self, logits, temperature, u, status=None, drafts=None, stream=None):
        """drafts [B, K] ~ softmax(logits / T) per row by inverse CDF with u [B, K]."""
        B, K, V = logits.shape
        dev = self.device
        _need(logits, torch.float32, dev, "logits")
        _need(u, torch.float32, dev, "u")
        if drafts is None:
            drafts = torch.empty(B, K, dtype=torch.int32, device=dev)
        _check(load().pe_sample_drafts(self._h, B, K, _p(logits), float(temperature), _p(u), _p(status), _p(drafts),
                                       _stream_ptr(stream)))
        return drafts

    def verify_stochastic(self, drafts, draft_logits, target_logits, temperature, u_accept, u_final, page_table,
                          num_pages, positions, seq_lens, stream=None):
        """Speculative-sampling acceptance + metadata rebuild. Returns a dict
        of int32 device tensors: accepted, final, emitted, positions,
        seq_lens, slot_mapping, rollback_slots, status."""
        B, K = drafts.shape
        dev = self.device
        for name, t in (("drafts", drafts), ("page_table", page_table), ("positions", positions),
                        ("seq_lens", seq_lens)):
            _need(t, torch.int32, dev, name)
        for name, t in (("draft_logits", draft_logits), ("target_logits", target_logits), ("u_accept", u_accept),
                        ("u_final", u_final)):
            _need(t, torch.float32, dev, name)
        e = lambda *s: torch.empty(*s, dtype=torch.int32, device=dev)
        o = dict(accepted=e(B), final=e(B), emitted=e(B, K + 1), positions=e(B), seq_lens=e(B),
                 slot_mapping=e(B, K), rollback_slots=e(B, K), status=e(B))
        _check(load().pe_verify_stochastic(
            self._h, B, K, _p(drafts), _p(draft_logits), _p(target_logits), float(temperature), _p(u_accept),
            _p(u_final), _p(page_table), page_table.shape[1], num_pages, _p(positions), _p(seq_lens),
            _p(o["positions"]), _p(o["seq_lens"]), _p(o["accepted"]), _p(o["final"]), _p(o["emitted"]),
            _p(o["slot_mapping"]), _p(o["rollback_slots"]), _p(o["status"]), _stream_ptr(stream)))
        return o

    def profile_start(self, kind, max_launches):
        """Time every launch of one kernel kind (name from KERNEL_KINDS) with
        CUDA events on its launch stream until profile_stop()."""
        _check(load().pe_profile_start(self._h, KERNEL_KINDS.index(kind), max_launches))

    def profile_stop(self):
        """(total device ms, launches timed) since profile_start()."""
        ms, n = ctypes.c_float(0), _i32(0)
        _check(load().pe_profile_stop(self._h, ctypes.byref(ms), ctypes.byref(n)))
        return ms.value, n.value

    def launch_count(self):
        return load().pe_last_launch_count(self._h)

    def test_stall_chain(self, stream=None):
        """Host-side fault injection (tests only): the next draft pass's
        layer-chain waits cannot complete and must give up."""
        _check(load().pe_test_stall_chain(self._h, _stream_ptr(stream)))

    def step_graph(self, last_token, target_hidden, positions, seq_lens, page_table, num_pages, k_cache, v_cache,
                   K, target_tokens, positions_out=None, seq_lens_out=None, sequential=False):
        """Capture draft + verify/rebuild into a replayable StepGraph over
        fixed buffers (outputs allocated here unless given)."""
        return StepGraph(self, last_token, target_hidden, positions, seq_lens, page_table, num_pages, k_cache,
                         v_cache, K, target_tokens, positions_out, seq_lens_out, sequential=sequential)

    def device_errors(self, stream=None):
        bits = ctypes.c_uint32(0)
        _check(load().pe_device_errors(self._h, _stream_ptr(stream), ctypes.byref(bits)))
        return bits.value

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            load().pe_destroy(self._h)
            self._h = _vp()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class StepGraph:
    """One draft pass + verify/rebuild captured into a CUDA graph by the
    library; ``launch()`` replays it. Buffers are fixed at capture."""

    def __init__(self, drafter, last_token, target_hidden, positions, seq_lens, page_table, num_pages, k_cache,
                 v_cache, K, target_tokens, positions_out=None, seq_lens_out=None, sequential=False):
        lib = load()
        dev = drafter.device
        B = last_token.shape[0]
        for name, t in (("last_token", last_token), ("positions", positions), ("seq_lens", seq_lens),
                        ("page_table", page_table), ("target_tokens", target_tokens)):
            _need(t, torch.int32, dev, name)
        _need(target_hidden, drafter.dtype, dev, "target_hidden")
        self.inputs = dict(last_token=last_token, target_hidden=target_hidden, positions=positions,
                           seq_lens=seq_lens, page_table=page_table, target_tokens=target_tokens,
                           k_cache=k_cache, v_cache=v_cache)
        # Every result the graph writes is a view into one int32 buffer
        # (`out_packed`, each view 64-byte aligned), so that a caller can read
        # all of a step's results back with a single copy.
        shapes = dict(drafts=(B, K), draft_status=(B,), accepted=(B,), bonus=(B,), emitted=(B, K + 1),
                      slot_mapping=(B, K), rollback_slots=(B, K), status=(B,))
        if positions_out is None:
            shapes["positions"] = (B,)
        if seq_lens_out is None:
            shapes["seq_lens"] = (B,)
        offs, total = {}, 0
        for name, shp in shapes.items():
            offs[name] = total
            n = 1
            for d in shp:
                n *= d
            total += (n + 15) // 16 * 16
        self.out_packed = torch.zeros(max(total, 16), dtype=torch.int32, device=dev)
        self.out = {}
        for name, shp in shapes.items():
            n = 1
            for d in shp:
                n *= d
            self.out[name] = self.out_packed.narrow(0, offs[name], n).view(*shp)
        if positions_out is not None:
            self.out["positions"] = positions_out
        if seq_lens_out is not None:
            self.out["seq_lens"] = seq_lens_out
        o = self.out
        g = _vp()
        _check(lib.pe_step_graph_create_ex(
            drafter._h, PE_DRAFT_SEQUENTIAL if sequential else PE_DRAFT_PARALLEL, B, K, _p(last_token), _p(target_hidden), _p(positions), _p(seq_lens), _p(page_table),
            page_table.shape[1], num_pages, _p(k_cache), _p(v_cache), _p(o["drafts"]), _p(o["draft_status"]),
            _p(target_tokens), _p(o["positions"]), _p(o["seq_lens"]), _p(o["accepted"]), _p(o["bonus"]),
            _p(o["emitted"]), _p(o["slot_mapping"]), _p(o["rollback_slots"]), _p(o["status"]), ctypes.byref(g)))
        self._g = g
        self._drafter = drafter     # keeps the handle (and its workspaces) alive

    def launch(self, stream=None):
        _check(load().pe_step_graph_launch(self._g, _stream_ptr(stream)))

    def launch_count(self):
        return load().pe_step_graph_launch_count(self._g)

    def close(self):
        if getattr(self, "_g", None) is not None and self._g.value:
            load().pe_step_graph_destroy(self._g)
            self._g = _vp()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def linear(w, x, stream=None):
    """y = x @ w.T in fp32 on the tcgen05 GEMM engine (bf16 or fp32/tf32 inputs)."""
    lib = load()
    M, Kd = w.shape
    N = x.shape[0]
    dtype = PE_DTYPE_BF16 if w.dtype == torch.bfloat16 else PE_DTYPE_FP32
    _need(x, w.dtype, w.device, "x")
    _need(w, w.dtype, w.device, "w")
    wsf, nt = ctypes.c_int64(0), _i32(0)
    _check(lib.pe_linear_scratch(dtype, M, N, Kd, ctypes.byref(wsf), ctypes.byref(nt)))
    ws = torch.empty(max(wsf.value, 1), dtype=torch.float32, device=w.device)
    tickets = torch.zeros(max(nt.value, 1), dtype=torch.int32, device=w.device)
    y = torch.empty(N, M, dtype=torch.float32, device=w.device)
    _check(lib.pe_linear(dtype, M, N, Kd, _p(w), _p(x), _p(y), _p(ws), _p(tickets), _stream_ptr(stream)))
    return y


def linear_fp8(w_codes, w_scale, x, stream=None):
    """y = x @ (decode(w_codes) * w_scale[:, None]).T in fp32: E4M3 weight
    codes (uint8 [M, Kd]), fp32 row scales [M], bf16 x [N, Kd]."""
    lib = load()
    M, Kd = w_codes.shape
    N = x.shape[0]
    _need(w_codes, torch.uint8, x.device, "w_codes")
    _need(w_scale, torch.float32, x.device, "w_scale")
    _need(x, torch.bfloat16, x.device, "x")
    wsf, nt = ctypes.c_int64(0), _i32(0)
    _check(lib.pe_linear_scratch(PE_DTYPE_FP8W, M, N, Kd, ctypes.byref(wsf), ctypes.byref(nt)))
    ws = torch.empty(max(wsf.value, 1), dtype=torch.float32, device=x.device)
    tickets = torch.zeros(max(nt.value, 1), dtype=torch.int32, device=x.device)
    y = torch.empty(N, M, dtype=torch.float32, device=x.device)
    _check(lib.pe_linear_fp8(M, N, Kd, _p(w_codes), _p(w_scale), _p(x), _p(y), _p(ws), _p(tickets),
                             _stream_ptr(stream)))
    return y


def linear_noalloc(w, x, y=None, stream=None):
    """y = x @ w.T through pe_linear_noalloc, which allocates no device memory
    (its split-K scratch is built into the library). Pass `y` to avoid the
    output allocation here as well."""
    lib = load()
    M, Kd = w.shape
    N = x.shape[0]
    dtype = PE_DTYPE_BF16 if w.dtype == torch.bfloat16 else PE_DTYPE_FP32
    _need(x, w.dtype, w.device, "x")
    _need(w, w.dtype, w.device, "w")
    if y is None:
        y = torch.empty(N, M, dtype=torch.float32, device=w.device)
    _need(y, torch.float32, w.device, "y")
    _check(lib.pe_linear_noalloc(dtype, M, N, Kd, _p(w), _p(x), _p(y), _stream_ptr(stream)))
    return y


def verify_rebuild(drafts, target_tokens, page_table, num_pages, positions, seq_lens, positions_out=None,
                   seq_lens_out=None, emitted=True, stream=None, out=None):
    """Greedy verify + metadata rebuild + rollback on the device.

    Returns a dict of int32 device tensors: accepted, bonus, emitted (or None),
    slot_mapping, rollback_slots, status, positions, seq_lens.
    """
    lib = load()
    B, K = drafts.shape
    dev = drafts.device
    for name, t in (("drafts", drafts), ("target_tokens", target_tokens), ("page_table", page_table),
                    ("positions", positions), ("seq_lens", seq_lens)):
        _need(t, torch.int32, dev, name)
    o = out if out is not None else {}

    def buf(name, *size):
        if name not in o or o[name] is None:
            o[name] = torch.empty(*size, dtype=torch.int32, device=dev)
        return o[name]

    pos_o = positions_out if positions_out is not None else buf("positions", B)
    sl_o = seq_lens_out if seq_lens_out is not None else buf("seq_lens", B)
    o["positions"], o["seq_lens"] = pos_o, sl_o
    em = buf("emitted", B, K + 1) if emitted else None
    _check(lib.pe_verify_rebuild(None, B, K, _p(drafts), _p(target_tokens), _p(page_table), page_table.shape[1],
                                 num_pages, _p(positions), _p(seq_lens), _p(pos_o), _p(sl_o),
                                 _p(buf("accepted", B)), _p(buf("bonus", B)), _p(em),
                                 _p(buf("slot_mapping", B, K)), _p(buf("rollback_slots", B, K)),
                                 _p(buf("status", B)), _stream_ptr(stream)))
    o["emitted"] = em
    return o


def verify_rebuild_refeed(drafts, target_tokens, page_table, num_pages, n_real, positions, seq_lens, stream=None):
    """Greedy verify + rebuild after a re-fed pass. Returns a dict of int32
    device tensors: accepted, bonus, emitted, n_real, positions, seq_lens,
    slot_mapping [B, 2K], rollback_slots [B, K], status."""
    lib = load()
    B, K = drafts.shape
    dev = drafts.device
    for name, t in (("drafts", drafts), ("target_tokens", target_tokens), ("page_table", page_table),
                    ("n_real", n_real), ("positions", positions), ("seq_lens", seq_lens)):
        _need(t, torch.int32, dev, name)
    e = lambda *s: torch.empty(*s, dtype=torch.int32, device=dev)
    o = dict(accepted=e(B), bonus=e(B), emitted=e(B, K + 1), n_real=e(B), positions=e(B), seq_lens=e(B),
             slot_mapping=e(B, 2 * K), rollback_slots=e(B, K), status=e(B))
    _check(lib.pe_verify_rebuild_refeed(None, B, K, _p(drafts), _p(target_tokens), _p(page_table),
                                        page_table.shape[1], num_pages, _p(n_real), _p(positions), _p(seq_lens),
                                        _p(o["n_real"]), _p(o["positions"]), _p(o["seq_lens"]), _p(o["accepted"]),
                                        _p(o["bonus"]), _p(o["emitted"]), _p(o["slot_mapping"]),
                                        _p(o["rollback_slots"]), _p(o["status"]), _stream_ptr(stream)))
    return o
