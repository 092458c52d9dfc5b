"""ctypes binding with the same names as the C ABI in ``include/mk.h``.

Argument marshalling only: the structs below mirror ``mk_config``,
``mk_layer_weights``, ``mk_weights``, ``mk_decode_opts`` and ``mk_info``; the
``Decoder`` class owns one ``mk_handle`` plus the torch device tensors whose
pointers the handle borrows.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional, Sequence

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))

MK_DECODE_PER_OP = 1
MK_DECODE_PER_OP_GRAPH = 2
MK_DECODE_STREAM = 4

_ERRORS = {0: "ok", -1: "invalid argument", -2: "unsupported shape or launch geometry",
           -3: "KV cache full", -4: "token id or sentinel row out of range",
           -5: "device wait timed out", -6: "non-finite logit", -7: "CUDA runtime error",
           -8: "device out of memory", -9: "position stream outside the rotary table"}


class MKError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__("%s: %s (%d)" % (what, _ERRORS.get(code, "unknown"), code))
        self.code = code


class mk_config(C.Structure):
    _fields_ = [("n_layers", C.c_int32), ("hidden", C.c_int32), ("n_q_heads", C.c_int32),
                ("n_kv_heads", C.c_int32), ("head_dim", C.c_int32), ("intermediate", C.c_int32),
                ("vocab", C.c_int32), ("vocab_in", C.c_int32), ("rms_eps", C.c_float),
                ("rope_theta", C.c_float), ("rope_mode", C.c_int32),
                ("mrope_sections", C.c_int32 * 3), ("max_seq", C.c_int32),
                ("rope_positions", C.c_int32), ("flags", C.c_uint32)]


class mk_layer_weights(C.Structure):
    _fields_ = [(k, C.c_void_p) for k in ("attn_norm", "wq", "wk", "wv", "q_norm", "k_norm", "wo",
                                          "mlp_norm", "w_gate", "w_up", "w_down")]


class mk_weights(C.Structure):
    _fields_ = [("embed", C.c_void_p), ("lm_head", C.c_void_p), ("final_norm", C.c_void_p),
                ("layers", C.POINTER(mk_layer_weights))]


class mk_decode_opts(C.Structure):
    _fields_ = [("flags", C.c_uint32), ("embeds", C.c_void_p), ("n_embed_rows", C.c_int32),
                ("pos3", C.c_void_p), ("logits", C.c_void_p), ("hidden", C.c_void_p),
                ("trace", C.c_void_p), ("attn_chunks", C.c_int32), ("spin_ns", C.c_int64),
                ("fault_skip_barrier", C.c_int32),
                ("books", C.c_void_p), ("n_books", C.c_int32), ("book_rows", C.c_int32),
                ("text", C.c_void_p), ("text_rows", C.c_int32), ("codes", C.c_void_p),
                ("text_ids", C.c_void_p), ("n_code_rows", C.c_int32)]


class mk_info(C.Structure):
    _fields_ = [("grid", C.c_int32), ("threads", C.c_int32), ("stages", C.c_int32),
                ("stage_bytes", C.c_int32), ("smem_bytes", C.c_int32), ("position", C.c_int32),
                ("max_chunks", C.c_int32), ("weight_bytes", C.c_int64), ("kv_bytes", C.c_int64),
                ("plan", C.c_int32)]


#: every symbol include/mk.h declares
EXPORTS = ("mk_create", "mk_reset_kv", "mk_decode", "mk_prefill", "mk_decode_start", "mk_decode_wait",
           "mk_mailbox_read", "mk_decode_host", "mk_get_info", "mk_embed_sum",
           "mk_embed_sum_noalloc", "mk_destroy", "mk_error_string", "mk_plan_for")

_lib = None


def lib_path() -> str:
    return os.path.join(_HERE, "libmk.so")


def load_library(path: Optional[str] = None):
    """Load libmk.so (in-tree) and declare the C signatures.  Raises if absent."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or lib_path()
    if not os.path.exists(p):
        raise RuntimeError("libmk.so not built at %s: run __graft_entry__.build()" % p)
    lib = C.CDLL(p)
    vp, i32, i64 = C.c_void_p, C.c_int32, C.c_int64
    lib.mk_create.argtypes = [C.POINTER(mk_config), C.POINTER(mk_weights), C.POINTER(vp)]
    lib.mk_reset_kv.argtypes = [vp, vp]
    lib.mk_decode.argtypes = [vp, vp, i32, i32, vp, C.POINTER(mk_decode_opts), vp]
    lib.mk_prefill.argtypes = [vp, vp, i32, vp, C.POINTER(mk_decode_opts), vp]
    lib.mk_decode_start.argtypes = [vp, vp, i32, i32, vp, C.POINTER(mk_decode_opts), vp]
    lib.mk_decode_wait.argtypes = [vp]
    lib.mk_mailbox_read.argtypes = [vp, vp, i32, C.POINTER(i32)]
    lib.mk_decode_host.argtypes = [vp, vp, i32, i32, vp, C.POINTER(mk_decode_opts), vp]
    lib.mk_get_info.argtypes = [vp, C.POINTER(mk_info)]
    lib.mk_plan_for.argtypes = [C.POINTER(mk_config), i32, C.POINTER(i32)]
    lib.mk_embed_sum.argtypes = [vp, i32, i32, vp, i32, i32, vp, vp, i32, vp, vp]
    lib.mk_embed_sum_noalloc.argtypes = [vp, i32, i32, vp, i32, i32, vp, vp, i32, vp, vp]
    lib.mk_destroy.argtypes = [vp]
    lib.mk_error_string.argtypes = [C.c_int]
    lib.mk_error_string.restype = C.c_char_p
    for name in EXPORTS:
        if name != "mk_error_string":
            getattr(lib, name).restype = C.c_int
    del i64
    if path is None:
        _lib = lib
    return lib


def error_string(code: int) -> str:
    return load_library().mk_error_string(code).decode()


def _check(rc: int, what: str):
    if rc != 0:
        raise MKError(rc, what)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream_ptr(stream) -> C.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def check_options(shape: dict, n: int, *, out=None, embeds=None, pos3=None, logits=None, hidden=None,
                  trace=None, grid: int = 0, talker=None, on_device: bool = True) -> None:
    """Validate the tensors of an ``n``-forward call against what the kernel
    reads and writes (the C ABI takes plain pointers and cannot check sizes):
    ``out`` int32 >= n ids; ``logits`` fp32 >= n x vocab; ``hidden`` fp32 >=
    n x (L + 1) x H; ``pos3`` int32 exactly 3 x n (three streams, row stride n);
    ``embeds`` fp32 [rows][H]; ``trace`` int64 >= n x (5 L + 1) x grid x 4;
    ``talker`` = (books bf16 [n_books][rows][H], text bf16 [rows][H], codes
    int32 [code_rows][n_books], text_ids int32 [code_rows]).  Every tensor must
    be contiguous (and on the device unless ``on_device`` is False).  Raises
    ValueError."""
    L, H, V = shape["n_layers"], shape["hidden"], shape["vocab"]

    def need(t, name, dtype, numel=None, exact=False, dims=None):
        if t is None:
            return
        if not isinstance(t, torch.Tensor) or t.dtype != dtype or not t.is_contiguous() or \
                (on_device and not t.is_cuda):
            raise ValueError("%s must be a contiguous device tensor of dtype %s" % (name, dtype))
        if dims is not None and t.dim() != dims:
            raise ValueError("%s must have %d dimensions" % (name, dims))
        if numel is not None and (t.numel() != numel if exact else t.numel() < numel):
            raise ValueError("%s holds %d elements; the call needs %s%d" %
                             (name, t.numel(), "" if exact else "at least ", numel))

    need(out, "out", torch.int32, n)
    need(logits, "logits", torch.float32, n * V)
    need(hidden, "hidden", torch.float32, n * (L + 1) * H)
    need(pos3, "pos3", torch.int32, 3 * n, exact=True)
    need(embeds, "embeds", torch.float32, dims=2)
    if embeds is not None and embeds.shape[1] != H:
        raise ValueError("embeds rows must have hidden (%d) elements" % H)
    if trace is not None:
        need(trace, "trace", torch.int64, n * (5 * L + 1) * grid * 4)
    if talker is not None:
        books, text, codes, text_ids = talker
        need(books, "talker books", torch.bfloat16, dims=3)
        need(text, "talker text", torch.bfloat16, dims=2)
        need(codes, "talker codes", torch.int32, dims=2)
        need(text_ids, "talker text_ids", torch.int32, codes.shape[0], exact=True)
        if books.shape[2] != H or text.shape[1] != H or codes.shape[1] != books.shape[0]:
            raise ValueError("talker tables must be [n_books][rows][H] and [rows][H], codes [rows][n_books]")


def check_embed_sum(books, text, codes, text_ids, out, on_device: bool = True) -> None:
    """Validate the tensors of ``mk_embed_sum`` / ``mk_embed_sum_noalloc``:
    books bf16 [n_books][rows][H], text bf16 [rows][H], codes int32 [n][n_books],
    text_ids int32 [n], out fp32 with at least n x H elements; all contiguous
    (and on the device unless ``on_device`` is False).  Raises ValueError."""
    if not isinstance(codes, torch.Tensor) or codes.dim() != 2:
        raise ValueError("codes must be a [n][n_books] int32 tensor")
    shape = dict(n_layers=0, hidden=books.shape[-1] if isinstance(books, torch.Tensor) and books.dim() == 3 else -1,
                 vocab=0)
    check_options(shape, codes.shape[0], talker=(books, text, codes, text_ids), on_device=on_device)
    n, H = codes.shape[0], books.shape[2]
    if not isinstance(out, torch.Tensor) or out.dtype != torch.float32 or not out.is_contiguous() or \
            (on_device and not out.is_cuda) or out.numel() < n * H:
        raise ValueError("out must be a contiguous fp32 %stensor of at least %d x %d elements"
                         % ("device " if on_device else "", n, H))


def check_weights(shape: dict, weights: dict, device=None) -> None:
    """Every weight must have the shape the config implies (``[out][in]``
    matrices, ``[n]`` gains); torch tensors must also be bf16, contiguous and
    on ``device``; numpy arrays must be uint16 bf16 bit patterns.  Raises
    ValueError (a wrong-sized matrix would otherwise be read past its end)."""
    s = shape
    H, L = s["hidden"], s["n_layers"]
    d, Hq, Hkv, I = s["head_dim"], s["n_q_heads"], s["n_kv_heads"], s["intermediate"]
    want = {"attn_norm": (H,), "wq": (Hq * d, H), "wk": (Hkv * d, H), "wv": (Hkv * d, H),
            "q_norm": (d,), "k_norm": (d,), "wo": (H, Hq * d), "mlp_norm": (H,),
            "w_gate": (I, H), "w_up": (I, H), "w_down": (H, I)}

    def one(a, name, shp):
        if isinstance(a, torch.Tensor):
            if a.dtype != torch.bfloat16 or not a.is_contiguous() or \
                    (device is not None and a.device != torch.device(device)):
                raise ValueError("weight %s must be a contiguous bf16 tensor on %s" % (name, device))
        elif isinstance(a, np.ndarray):
            if a.dtype != np.uint16:
                raise ValueError("weight %s must hold bf16 bit patterns (uint16)" % name)
        else:
            raise ValueError("weight %s must be a torch tensor or a numpy array" % name)
        if tuple(a.shape) != tuple(shp):
            raise ValueError("weight %s has shape %s; the config needs %s" % (name, tuple(a.shape), tuple(shp)))

    one(weights["embed"], "embed", (s["vocab_in"], H))
    one(weights["final_norm"], "final_norm", (H,))
    if weights.get("lm_head") is not None:
        one(weights["lm_head"], "lm_head", (s["vocab"], H))
    elif s["vocab"] != s["vocab_in"]:
        raise ValueError("a tied head needs vocab == vocab_in")
    if len(weights["layers"]) != L:
        raise ValueError("%d layers given; the config has %d" % (len(weights["layers"]), L))
    for l, lw in enumerate(weights["layers"]):
        for k, shp in want.items():
            one(lw[k], "layers[%d].%s" % (l, k), shp)


def config_struct(s: dict, max_seq: int, rope_positions: int = 0) -> mk_config:
    """The ``mk_config`` of a shape dict (``workloads.shape``)."""
    cfg = mk_config()
    cfg.n_layers, cfg.hidden = s["n_layers"], s["hidden"]
    cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim = s["n_q_heads"], s["n_kv_heads"], s["head_dim"]
    cfg.intermediate, cfg.vocab, cfg.vocab_in = s["intermediate"], s["vocab"], s["vocab_in"]
    cfg.rms_eps, cfg.rope_theta = s.get("rms_eps", 1e-6), s.get("rope_theta", 1e6)
    ms = s.get("mrope_sections")
    cfg.rope_mode = 0 if ms is None else (2 if s.get("mrope_interleaved") else 1)
    if ms is not None:
        cfg.mrope_sections[0], cfg.mrope_sections[1], cfg.mrope_sections[2] = ms
    cfg.max_seq, cfg.rope_positions, cfg.flags = max_seq, rope_positions, 0
    return cfg


def plan_for(s: dict, n_sm: int, max_seq: int = 4096) -> int:
    """``mk_plan_for``: the decode kernel mk_create picks for shape ``s`` on a
    device with ``n_sm`` multiprocessors (0 general, 1 / 2 the kernels compiled
    for the 0.6B / 1.7B dims).  Needs no device."""
    lib = load_library()
    plan = C.c_int32(-1)
    _check(lib.mk_plan_for(C.byref(config_struct(s, max_seq)), int(n_sm), C.byref(plan)), "mk_plan_for")
    return plan.value


def _dev_bf16(bits: np.ndarray, device) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to(device, non_blocking=False).contiguous()


def _require_cuda():
    if not torch.cuda.is_available():
        raise RuntimeError("persistent_transformer_megakernel_gb300 needs a CUDA device (GB300)")


class Decoder:
    """One decode session: weights on the device, a KV cache, a cursor.

    ``shape`` is a dict (see ``workloads.SHAPES``); ``weights`` holds bf16 bit
    patterns as numpy ``uint16`` arrays (``workloads.make_weights``) or torch
    bf16 tensors already on the device."""

    def __init__(self, shape: dict, weights: dict, max_seq: int, rope_positions: int = 0,
                 device="cuda:0"):
        _require_cuda()
        self.lib = load_library()
        self.device = torch.device(device)
        torch.cuda.set_device(self.device)
        self.shape = dict(shape)
        s = self.shape
        check_weights(s, weights, self.device if isinstance(weights["embed"], torch.Tensor) else None)
        conv = (lambda a: a) if isinstance(weights["embed"], torch.Tensor) else \
            (lambda a: _dev_bf16(a, self.device))
        self._keep = []

        def dev(a):
            t = conv(a)
            self._keep.append(t)
            return t

        self.embed = dev(weights["embed"])
        self.final_norm = dev(weights["final_norm"])
        self.lm_head = None if weights.get("lm_head") is None else dev(weights["lm_head"])
        L = s["n_layers"]
        self._layers = (mk_layer_weights * L)()
        for l, lw in enumerate(weights["layers"]):
            for k in mk_layer_weights._fields_:
                setattr(self._layers[l], k[0], dev(lw[k[0]]).data_ptr())
        cfg = config_struct(s, max_seq, rope_positions)
        w = mk_weights()
        w.embed = self.embed.data_ptr()
        w.lm_head = None if self.lm_head is None else self.lm_head.data_ptr()
        w.final_norm = self.final_norm.data_ptr()
        w.layers = self._layers
        h = C.c_void_p()
        _check(self.lib.mk_create(C.byref(cfg), C.byref(w), C.byref(h)), "mk_create")
        self.h = h
        self.max_seq = max_seq
        self._out = torch.empty(max_seq, dtype=torch.int32, device=self.device)

    # ---------------------------------------------------------------- basics
    def info(self) -> dict:
        i = mk_info()
        _check(self.lib.mk_get_info(self.h, C.byref(i)), "mk_get_info")
        return {k: getattr(i, k) for k, _ in mk_info._fields_}

    @property
    def position(self) -> int:
        return self.info()["position"]

    def reset(self, stream=None):
        _check(self.lib.mk_reset_kv(self.h, _stream_ptr(stream)), "mk_reset_kv")

    def close(self):
        if getattr(self, "h", None):
            self.lib.mk_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ---------------------------------------------------------------- decode
    def _opts(self, per_op, embeds, pos3, logits, hidden, trace, attn_chunks, spin_ns,
              fault_skip_barrier, talker=None):
        o = mk_decode_opts()
        o.flags = (MK_DECODE_PER_OP_GRAPH if per_op == "graph" else MK_DECODE_PER_OP) if per_op else 0
        o.embeds = _ptr(embeds)
        o.n_embed_rows = 0 if embeds is None else embeds.shape[0]
        o.pos3 = _ptr(pos3)
        o.logits = _ptr(logits)
        o.hidden = _ptr(hidden)
        o.trace = _ptr(trace)
        o.attn_chunks = attn_chunks
        o.spin_ns = spin_ns
        o.fault_skip_barrier = fault_skip_barrier
        if talker is not None:
            # (books bf16 [n_books][rows][H], text bf16 [rows][H], codes int32 [n][n_books], text_ids int32 [n])
            books, text, codes, text_ids = talker
            o.books = _ptr(books)
            o.n_books, o.book_rows = books.shape[0], books.shape[1]
            o.text = _ptr(text)
            o.text_rows = text.shape[0]
            o.codes = _ptr(codes)
            o.text_ids = _ptr(text_ids)
            o.n_code_rows = codes.shape[0]
        return o

    def decode(self, in_ids=None, n_steps: int = 0, *, out: Optional[torch.Tensor] = None,
               per_op=False, embeds: Optional[torch.Tensor] = None,
               pos3: Optional[torch.Tensor] = None, logits: Optional[torch.Tensor] = None,
               hidden: Optional[torch.Tensor] = None, trace: Optional[torch.Tensor] = None,
               attn_chunks: int = 0, spin_ns: int = 0, fault_skip_barrier: int = 0,
               talker=None, stream=None) -> torch.Tensor:
        """``mk_decode``: ``in_ids`` (device int32 tensor, or a sequence moved to
        the device) then ``n_steps`` greedy forwards.  Returns the ids tensor.
        ``per_op=True`` runs the one-launch-per-phase ablation, ``per_op="graph"``
        the same launches replayed from a captured CUDA graph.  ``talker`` =
        ``(books, text, codes, text_ids)`` device tensors: negative ids select code
        rows whose codebook + text sum the kernel forms itself."""
        if in_ids is None:
            d_in = None
            n_in = 0
        else:
            d_in = in_ids if isinstance(in_ids, torch.Tensor) else \
                torch.as_tensor(np.asarray(in_ids, dtype=np.int32), device=self.device)
            d_in = d_in.to(device=self.device, dtype=torch.int32).contiguous()
            n_in = d_in.numel()
        n = n_in + n_steps
        if out is None:
            out = torch.empty(max(n, 1), dtype=torch.int32, device=self.device)
        check_options(self.shape, n, out=out, embeds=embeds, pos3=pos3, logits=logits, hidden=hidden,
                      trace=trace, grid=self.info()["grid"] if trace is not None else 0, talker=talker)
        o = self._opts(per_op, embeds, pos3, logits, hidden, trace, attn_chunks, spin_ns,
                       fault_skip_barrier, talker)
        rc = self.lib.mk_decode(self.h, _ptr(d_in), n_in, n_steps, _ptr(out), C.byref(o),
                                _stream_ptr(stream))
        _check(rc, "mk_decode")
        return out[:n]

    def prefill(self, in_ids, *, out: Optional[torch.Tensor] = None, all_ids: bool = True,
                embeds: Optional[torch.Tensor] = None, pos3: Optional[torch.Tensor] = None,
                logits: Optional[torch.Tensor] = None, hidden: Optional[torch.Tensor] = None,
                stream=None) -> Optional[torch.Tensor]:
        """``mk_prefill``: the prompt's forwards as batched tensor-core GEMMs.
        Returns the greedy id after every prompt token (``all_ids``) or None
        (then only the last token's logits are computed; the next ``decode``
        continues from its id)."""
        d_in = in_ids if isinstance(in_ids, torch.Tensor) else \
            torch.as_tensor(np.asarray(in_ids, dtype=np.int32), device=self.device)
        d_in = d_in.to(device=self.device, dtype=torch.int32).contiguous()
        n = d_in.numel()
        if all_ids and out is None:
            out = torch.empty(max(n, 1), dtype=torch.int32, device=self.device)
        check_options(self.shape, n, out=out if all_ids else None, embeds=embeds, pos3=pos3, logits=logits,
                      hidden=hidden)
        o = self._opts(False, embeds, pos3, logits, hidden, None, 0, 0, 0)
        _check(self.lib.mk_prefill(self.h, _ptr(d_in), n, _ptr(out) if all_ids else None, C.byref(o),
                                   _stream_ptr(stream)), "mk_prefill")
        return out[:n] if all_ids else None

    def decode_start(self, in_ids=None, n_steps: int = 0, *, out: Optional[torch.Tensor] = None,
                     stream_ids: bool = True, per_op=False, embeds: Optional[torch.Tensor] = None,
                     pos3: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        """``mk_decode_start``: enqueue the decode and return at once (with
        ``stream_ids`` every greedy id is published to the host mailbox as it
        is chosen).  ``decode_wait`` must follow.  Returns the device ids tensor
        that holds all ids once the wait has returned."""
        if in_ids is None:
            d_in, n_in = None, 0
        else:
            d_in = in_ids if isinstance(in_ids, torch.Tensor) else \
                torch.as_tensor(np.asarray(in_ids, dtype=np.int32), device=self.device)
            d_in = d_in.to(device=self.device, dtype=torch.int32).contiguous()
            n_in = d_in.numel()
        n = n_in + n_steps
        if out is None:
            out = torch.empty(max(n, 1), dtype=torch.int32, device=self.device)
        check_options(self.shape, n, out=out, embeds=embeds, pos3=pos3)
        o = self._opts(per_op, embeds, pos3, None, None, None, 0, 0, 0)
        if stream_ids:
            o.flags |= MK_DECODE_STREAM
        self._pending_keep = (d_in, out, embeds, pos3)   # alive until the wait
        _check(self.lib.mk_decode_start(self.h, _ptr(d_in), n_in, n_steps, _ptr(out), C.byref(o),
                                        _stream_ptr(stream)), "mk_decode_start")
        return out[:n]

    def decode_wait(self) -> None:
        """``mk_decode_wait``: the status of the started decode."""
        rc = self.lib.mk_decode_wait(self.h)
        self._pending_keep = None
        _check(rc, "mk_decode_wait")

    def mailbox(self, cap: int = None) -> np.ndarray:
        """``mk_mailbox_read``: the ids the streaming decode has published so far."""
        cap = self.max_seq if cap is None else cap
        buf = np.empty(max(cap, 1), dtype=np.int32)
        n = C.c_int32(0)
        _check(self.lib.mk_mailbox_read(self.h, buf.ctypes.data_as(C.c_void_p), cap, C.byref(n)),
               "mk_mailbox_read")
        return buf[:min(n.value, cap)].copy()

    def decode_stream(self, in_ids=None, n_steps: int = 0, *, timeout_s: float = 60.0, **kw):
        """Generator over ``(i, id, t)`` for every forward of a streaming
        decode, in order, as the host sees each id appear (``t`` seconds after
        the launch was enqueued).  The decode is waited for at the end."""
        import time
        n_in = 0 if in_ids is None else len(in_ids)
        n = n_in + n_steps
        t0 = time.perf_counter()
        self.decode_start(in_ids, n_steps, stream_ids=True, **kw)
        seen = 0
        try:
            while seen < n:
                ids = self.mailbox(n)
                now = time.perf_counter() - t0
                for i in range(seen, len(ids)):
                    yield i, int(ids[i]), now
                seen = max(seen, len(ids))
                if seen < n and torch.cuda.current_stream(self.device).query() and \
                        len(self.mailbox(n)) == seen:
                    break            # the launch ended early (an error): the wait reports it
                if seen < n and now > timeout_s:
                    raise RuntimeError("streaming decode: only %d of %d ids after %.0f s" % (seen, n, now))
        finally:
            self.decode_wait()

    def decode_host(self, in_ids: Sequence[int], n_steps: int = 0, *, per_op: bool = False,
                    embeds=None, pos3=None, stream=None) -> np.ndarray:
        """``mk_decode_host``: host id buffers in and out (the copies are part of the call)."""
        ids = np.ascontiguousarray(np.asarray(in_ids, dtype=np.int32))
        n = ids.size + n_steps
        out = np.empty(max(n, 1), dtype=np.int32)
        check_options(self.shape, n, embeds=embeds, pos3=pos3)
        o = self._opts(per_op, embeds, pos3, None, None, None, 0, 0, 0)
        rc = self.lib.mk_decode_host(self.h, ids.ctypes.data_as(C.c_void_p) if ids.size else None,
                                     ids.size, n_steps, out.ctypes.data_as(C.c_void_p), C.byref(o),
                                     _stream_ptr(stream))
        _check(rc, "mk_decode_host")
        return out[:n]


def embed_sum(books: torch.Tensor, text: torch.Tensor, codes: torch.Tensor, text_ids: torch.Tensor,
              out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """``mk_embed_sum``: per-step sum of codebook rows and a text row (fp32)."""
    _require_cuda()
    lib = load_library()
    n_books, book_rows, H = books.shape
    n = codes.shape[0]
    if out is None:
        out = torch.empty((n, H), dtype=torch.float32, device=books.device)
    codes_i = codes.to(torch.int32).contiguous()
    text_i = text_ids.to(torch.int32).contiguous()
    check_embed_sum(books, text, codes_i, text_i, out)
    rc = lib.mk_embed_sum(_ptr(books), n_books, book_rows, _ptr(text), text.shape[0], H,
                          _ptr(codes_i), _ptr(text_i), n, _ptr(out), _stream_ptr(stream))
    _check(rc, "mk_embed_sum")
    return out


def embed_sum_noalloc(books: torch.Tensor, text: torch.Tensor, codes: torch.Tensor, text_ids: torch.Tensor,
                      out: torch.Tensor, stream=None) -> torch.Tensor:
    """``mk_embed_sum_noalloc``: the same rows as ``embed_sum`` into a caller
    buffer, with the library's static scratch (at most 4096 rows a call); the
    library allocates nothing.  ``out`` is required (fp32, >= n x H)."""
    _require_cuda()
    lib = load_library()
    check_embed_sum(books, text, codes, text_ids, out)
    n_books, book_rows, H = books.shape
    rc = lib.mk_embed_sum_noalloc(_ptr(books), n_books, book_rows, _ptr(text), text.shape[0], H, _ptr(codes),
                                  _ptr(text_ids), codes.shape[0], _ptr(out), _stream_ptr(stream))
    _check(rc, "mk_embed_sum_noalloc")
    return out
