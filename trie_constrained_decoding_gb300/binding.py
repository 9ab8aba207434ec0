"""Thin ctypes binding over ``libtcd.so`` (the C ABI of ``include/tcd.h``).

Argument marshalling only: every step of the decode path runs in the CUDA
kernels behind the C ABI.  Device buffers are passed as torch CUDA tensors
(their ``data_ptr()``), streams as ``torch.cuda.Stream`` (default: the current
stream).  If the library is missing this module raises on import; there is no
CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.environ.get("TCD_LIB", os.path.join(_HERE, "libtcd.so"))

if not os.path.exists(LIB_PATH):
    raise ImportError(f"libtcd.so not found at {LIB_PATH}: build it with "
                      "`python -m trie_constrained_decoding_gb300.build` (no CPU fallback exists)")

_lib = ctypes.CDLL(LIB_PATH)

# Status codes and enums of include/tcd.h
TC_OK = 0
STATUS_NAMES = {}
RES_AUTO, RES_CONST, RES_GLOBAL = 0, 1, 2
BIND_LIVE_COUNTS = 0x10        # or-ed into bind's residency: per-sequence live-count arrays for every k
HEAD_SPARSE, HEAD_DENSE, HEAD_UNION_GEMM, HEAD_DENSE_GEMM = 0, 1, 2, 3
FLAG_JUMP_FORWARD = 0x100      # or-ed into `head` of decode / decode_graph: forced tokens skip the head
FLAG_FORCED_LOGITS = 0x200     # with FLAG_JUMP_FORWARD: forced tokens still get their logits
FLAG_ROOT_GEMM = 0x400         # with HEAD_SPARSE in decodes: the first (root) step on the tcgen05 GEMM
STAT_SLOTS = 6
TC_ERR_EMPTY_MASK, TC_ERR_NO_LIVE_EDGE, TC_ERR_MAX_STEPS, TC_ERR_BOUNDS = 16, 17, 18, 19
TC_ERR_DEVICE_TIMEOUT = 20
CONST_CAPACITY_BYTES = 63 * 1024

_i32p = ctypes.POINTER(ctypes.c_int32)
_i64p = ctypes.POINTER(ctypes.c_int64)
_vp = ctypes.c_void_p


class _TrieInfo(ctypes.Structure):
    _fields_ = [("n_nodes", ctypes.c_int32), ("n_edges", ctypes.c_int32), ("n_strings", ctypes.c_int32),
                ("max_fanout", ctypes.c_int32), ("root_fanout", ctypes.c_int32), ("max_depth", ctypes.c_int32),
                ("vocab", ctypes.c_int32), ("sep_id", ctypes.c_int32), ("stop_id", ctypes.c_int32),
                ("header_bytes", ctypes.c_int32), ("total_tokens", ctypes.c_int64),
                ("walk_image_bytes", ctypes.c_int64)]


class Sampling(ctypes.Structure):
    """tc_sampling_t: temperature > 0, top_k >= 0 (0: off), top_p in [0, 1] (1: off)."""
    _fields_ = [("temperature", ctypes.c_float), ("top_k", ctypes.c_int32), ("top_p", ctypes.c_float)]


def _decl(name, restype, argtypes):
    f = getattr(_lib, name)
    f.restype = restype
    f.argtypes = argtypes
    return f


_compile = _decl("tc_compile_trie", ctypes.c_int, [_i32p, _i64p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                                   ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(_vp)])
_compile_chars = _decl("tc_compile_char_trie", ctypes.c_int,
                       [_vp, _i64p, ctypes.c_int32, _i32p, _vp, _i64p, ctypes.c_int32, ctypes.c_int32,
                        ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(_vp)])
_info = _decl("tc_trie_info", ctypes.c_int, [_vp, ctypes.POINTER(_TrieInfo)])
_export = _decl("tc_trie_export", ctypes.c_int, [_vp] + [_i32p] * 7)
_trie_free = _decl("tc_trie_free", None, [_vp])
_export_ranks = _decl("tc_trie_export_ranks", ctypes.c_int, [_vp, _i32p, _i32p])
_ctx_create = _decl("tc_ctx_create", ctypes.c_int, [ctypes.c_int32, _vp, ctypes.c_int32, ctypes.c_int32,
                                                   ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(_vp)])
_ctx_destroy = _decl("tc_ctx_destroy", None, [_vp])
_bind = _decl("tc_bind_grammar", ctypes.c_int, [_vp, _vp, ctypes.c_int32, _vp])
_bound_res = _decl("tc_bound_residency", ctypes.c_int, [_vp, _i32p])
_reset = _decl("tc_reset", ctypes.c_int, [_vp, ctypes.c_int32, ctypes.c_int32, _vp])
_step = _decl("tc_step", ctypes.c_int, [_vp, _vp, ctypes.c_int32, _vp, _vp, _vp, _vp])
_decode_args = [_vp, _vp, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                _vp, _vp, _vp, _vp]
_decode = _decl("tc_decode", ctypes.c_int, _decode_args + [_vp])
_decode_host = _decl("tc_decode_host", ctypes.c_int, _decode_args + [_vp])
_graph_create = _decl("tc_decode_graph_create", ctypes.c_int, _decode_args + [ctypes.POINTER(_vp)])
_graph_launch = _decl("tc_graph_launch", ctypes.c_int, [_vp, _vp])
_graph_destroy = _decl("tc_graph_destroy", None, [_vp])
_first_error = _decl("tc_first_error", ctypes.c_int, [_vp, _vp, _i32p, _i32p])
_read_state = _decl("tc_read_seq_state", ctypes.c_int, [_vp, _vp] + [_i32p] * 5)
_read_stats = _decl("tc_read_stats", ctypes.c_int, [_vp, _vp, _i64p, ctypes.c_int32])
_decode_sample = _decl("tc_decode_sample", ctypes.c_int,
                       [_vp, _vp, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                        ctypes.POINTER(Sampling), _vp, _vp, _vp, _vp, _vp, _vp])
_step_sample = _decl("tc_step_sample", ctypes.c_int, [_vp, _vp, ctypes.c_int32, ctypes.POINTER(Sampling), _vp, _vp,
                                                      _vp, _vp, _vp])
_loop_floor = _decl("tc_loop_floor", ctypes.c_int, [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _vp,
                                                    ctypes.POINTER(ctypes.c_float), _i64p])
_gemm_wait_test = _decl("tc_gemm_wait_test", ctypes.c_int, [_vp, ctypes.c_int32, ctypes.c_int64])
_status_str = _decl("tc_status_str", ctypes.c_char_p, [ctypes.c_int])
_last_msg = _decl("tc_last_error_message", ctypes.c_char_p, [])


def status_name(code: int) -> str:
    return _status_str(int(code)).decode()


class TcError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = int(code)
        self.name = status_name(code)
        msg = _last_msg().decode()
        super().__init__(f"{where}: {self.name}" + (f" ({msg})" if msg else ""))


def _check(code: int, where: str):
    if code != TC_OK:
        raise TcError(code, where)


def _stream_ptr(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


class Trie:
    """A compiled catalog (host object)."""

    def __init__(self, handle):
        self._h = handle

    @classmethod
    def compile(cls, catalog: Sequence[Sequence[int]], sep_id: int, stop_id: int, vocab: int,
                max_fanout: int = 256) -> "Trie":
        lens = [len(s) for s in catalog]
        offsets = np.zeros(len(catalog) + 1, dtype=np.int64)
        offsets[1:] = np.cumsum(lens)
        ids = np.array([t for s in catalog for t in s], dtype=np.int32) if offsets[-1] else np.zeros(1, np.int32)
        h = _vp()
        code = _compile(ids.ctypes.data_as(_i32p), offsets.ctypes.data_as(_i64p), len(catalog), sep_id, stop_id,
                        vocab, max_fanout, ctypes.byref(h))
        _check(code, "tc_compile_trie")
        return cls(h)

    @classmethod
    def compile_chars(cls, strings: Sequence[bytes], vocab: Sequence[tuple], sep_id: int, stop_id: int,
                      vocab_size: int, max_fanout: int = 4096) -> "Trie":
        """tc_compile_char_trie: byte strings and a byte vocabulary [(token id, bytes)]."""
        offs = np.zeros(len(strings) + 1, dtype=np.int64)
        offs[1:] = np.cumsum([len(x) for x in strings])
        chars = np.frombuffer(b"".join(strings), dtype=np.uint8).copy()
        ids = np.array([i for i, _ in vocab], dtype=np.int32)
        toff = np.zeros(len(vocab) + 1, dtype=np.int64)
        toff[1:] = np.cumsum([len(b) for _, b in vocab])
        tchars = np.frombuffer(b"".join(b for _, b in vocab), dtype=np.uint8).copy()
        h = _vp()
        code = _compile_chars(chars.ctypes.data, offs.ctypes.data_as(_i64p), len(strings),
                              ids.ctypes.data_as(_i32p), tchars.ctypes.data, toff.ctypes.data_as(_i64p), len(vocab),
                              sep_id, stop_id, vocab_size, max_fanout, ctypes.byref(h))
        _check(code, "tc_compile_char_trie")
        return cls(h)

    def info(self) -> dict:
        inf = _TrieInfo()
        _check(_info(self._h, ctypes.byref(inf)), "tc_trie_info")
        return {name: getattr(inf, name) for name, _ in _TrieInfo._fields_}

    def export(self) -> dict:
        i = self.info()
        N, E, K, T = i["n_nodes"], i["n_edges"], i["n_strings"], i["total_tokens"]
        arrs = {"node_begin": N + 1, "edge_tok": E, "edge_child": E, "node_ptr": N, "static_cnt": E,
                "path_off": K + 1, "path": max(T, 1)}
        out = {k: np.zeros(n, dtype=np.int32) for k, n in arrs.items()}
        _check(_export(self._h, *[out[k].ctypes.data_as(_i32p) for k in arrs]), "tc_trie_export")
        out["path"] = out["path"][:T]
        return out

    def ranks(self) -> dict:
        """Depth-first pointer ranks (tc_trie_export_ranks): ptr_rank[K], edge_lo[E]."""
        i = self.info()
        out = {"ptr_rank": np.zeros(i["n_strings"], dtype=np.int32), "edge_lo": np.zeros(i["n_edges"], np.int32)}
        _check(_export_ranks(self._h, out["ptr_rank"].ctypes.data_as(_i32p), out["edge_lo"].ctypes.data_as(_i32p)),
               "tc_trie_export_ranks")
        return out

    def close(self):
        if self._h:
            _trie_free(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Graph:
    def __init__(self, ctx, handle, keep):
        self._ctx, self._h, self._keep = ctx, handle, keep

    def launch(self, stream=None):
        _check(_graph_launch(self._h, _stream_ptr(stream)), "tc_graph_launch")

    def close(self):
        if self._h:
            _graph_destroy(self._h)
            self._h = None


class Context:
    """A decoding context over a bf16 tied embedding held in a torch CUDA tensor."""

    def __init__(self, emb, max_batch: int, cand_cap: int = 256, device: Optional[int] = None):
        import torch
        if not (emb.is_cuda and emb.dtype == torch.bfloat16 and emb.dim() == 2 and emb.is_contiguous()):
            raise ValueError("emb must be a contiguous 2-D bfloat16 CUDA tensor [vocab, hidden]")
        self.emb = emb                   # keep the embedding alive
        self.vocab, self.hidden = emb.shape
        self.device = emb.device.index if device is None else device
        self.max_batch = max_batch
        h = _vp()
        _check(_ctx_create(self.device, emb.data_ptr(), self.vocab, self.hidden, max_batch, cand_cap,
                           ctypes.byref(h)), "tc_ctx_create")
        self._h = h
        self._graphs = []

    def bind(self, trie: Trie, residency: int = RES_AUTO, stream=None):
        _check(_bind(self._h, trie._h, residency, _stream_ptr(stream)), "tc_bind_grammar")

    def residency(self) -> int:
        r = ctypes.c_int32()
        _check(_bound_res(self._h, ctypes.byref(r)), "tc_bound_residency")
        return r.value

    def reset(self, batch: int, k: int, stream=None):
        _check(_reset(self._h, batch, k, _stream_ptr(stream)), "tc_reset")

    def step(self, hidden, tok_out, logit_out=None, status_out=None, head: int = HEAD_SPARSE, stream=None):
        _check(_step(self._h, hidden.data_ptr(), head, tok_out.data_ptr(), _ptr(logit_out), _ptr(status_out),
                     _stream_ptr(stream)), "tc_step")

    def _dargs(self, hidden_steps, k, max_steps, head, toks, logits, lens, status):
        S, B, H = hidden_steps.shape
        return (self._h, hidden_steps.data_ptr(), S, B, k, max_steps, head, toks.data_ptr(), logits.data_ptr(),
                lens.data_ptr(), status.data_ptr())

    def decode(self, hidden_steps, k, max_steps, toks, logits, lens, status, head=HEAD_SPARSE, stream=None):
        _check(_decode(*self._dargs(hidden_steps, k, max_steps, head, toks, logits, lens, status),
                       _stream_ptr(stream)), "tc_decode")

    def decode_sample(self, hidden_steps, k, max_steps, uniforms, toks, logits, lens, status, temperature=1.0,
                      top_k=0, top_p=1.0, head=HEAD_SPARSE, stream=None):
        """tc_decode_sample: uniforms is a device float32 [batch, max_steps] tensor."""
        S, B, H = hidden_steps.shape
        sp = Sampling(float(temperature), int(top_k), float(top_p))
        _check(_decode_sample(self._h, hidden_steps.data_ptr(), S, B, k, max_steps, head, ctypes.byref(sp),
                              uniforms.data_ptr(), toks.data_ptr(), logits.data_ptr(), lens.data_ptr(),
                              status.data_ptr(), _stream_ptr(stream)), "tc_decode_sample")

    def step_sample(self, hidden, uniforms, tok_out, logit_out=None, status_out=None, temperature=1.0, top_k=0,
                    top_p=1.0, head: int = HEAD_SPARSE, stream=None):
        sp = Sampling(float(temperature), int(top_k), float(top_p))
        _check(_step_sample(self._h, hidden.data_ptr(), head, ctypes.byref(sp), uniforms.data_ptr(),
                            tok_out.data_ptr(), _ptr(logit_out), _ptr(status_out), _stream_ptr(stream)),
               "tc_step_sample")

    def decode_host(self, hidden_steps, k, max_steps, toks, logits, lens, status, head=HEAD_SPARSE, stream=None):
        _check(_decode_host(*self._dargs(hidden_steps, k, max_steps, head, toks, logits, lens, status),
                            _stream_ptr(stream)), "tc_decode_host")

    def decode_graph(self, hidden_steps, k, max_steps, toks, logits, lens, status, head=HEAD_SPARSE) -> Graph:
        h = _vp()
        _check(_graph_create(*self._dargs(hidden_steps, k, max_steps, head, toks, logits, lens, status),
                             ctypes.byref(h)), "tc_decode_graph_create")
        g = Graph(self, h, (hidden_steps, toks, logits, lens, status))
        self._graphs.append(g)
        return g

    def first_error(self, stream=None):
        seq, code = ctypes.c_int32(), ctypes.c_int32()
        _check(_first_error(self._h, _stream_ptr(stream), ctypes.byref(seq), ctypes.byref(code)), "tc_first_error")
        return seq.value, code.value

    def raise_on_error(self, stream=None):
        seq, code = self.first_error(stream)
        if code != TC_OK:
            raise TcError(code, f"sequence {seq}")

    def seq_state(self, batch: int, stream=None) -> dict:
        out = {k: np.zeros(batch, dtype=np.int32) for k in ("node", "emitted", "len", "status", "done")}
        _check(_read_state(self._h, _stream_ptr(stream), *[out[k].ctypes.data_as(_i32p) for k in
                                                           ("node", "emitted", "len", "status", "done")]),
               "tc_read_seq_state")
        return out

    def stats(self, reset: bool = False, stream=None) -> dict:
        out = np.zeros(STAT_SLOTS, dtype=np.int64)
        _check(_read_stats(self._h, _stream_ptr(stream), out.ctypes.data_as(_i64p), int(reset)), "tc_read_stats")
        return {"step_launches": int(out[0]), "seq_steps": int(out[1]), "cand_rows": int(out[2]),
                "reset_launches": int(out[3]), "forced": int(out[4]), "union_rows": int(out[5])}

    def gemm_wait_test(self, withhold: bool, wait_polls: int = 0):
        """tc_gemm_wait_test: make the GEMM heads' first pipeline stage never
        arrive (withhold) with waits of `wait_polls` polls; (False, 0) restores."""
        _check(_gemm_wait_test(self._h, int(bool(withhold)), int(wait_polls)), "tc_gemm_wait_test")

    def close(self):
        for g in self._graphs:
            g.close()
        self._graphs = []
        if self._h:
            _ctx_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def loop_floor(device: int, batch: int, iterations: int, stream=None):
    """Milliseconds and kernel launches of the decode loop's graph shape with
    do-nothing kernels in the steps' place (tc_loop_floor)."""
    ms = ctypes.c_float()
    n = ctypes.c_int64()
    _check(_loop_floor(device, batch, iterations, _stream_ptr(stream), ctypes.byref(ms), ctypes.byref(n)),
           "tc_loop_floor")
    return float(ms.value), int(n.value)
