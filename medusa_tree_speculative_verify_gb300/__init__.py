"""Python binding of libmedusa_verify.so: argument marshalling only.

Every entry point has the name of its C function (see include/medusa_verify.h)
and passes torch tensors as raw device pointers on the current CUDA stream.
All computation happens in the library's kernels; if the library is missing
or fails to load, :func:`lib` raises -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from .build import LIB, build

__all__ = ["lib", "MVError", "Tree", "AcceptParams", "PosteriorResult", "GREEDY", "TYPICAL", "Model", "Session",
           "RootParams", "ROOT_ARGMAX", "ROOT_TYPICAL", "ROOT_NUCLEUS", "sample_root",
           "linear_bf16", "linear_bf16_workspace", "ModelDims",
           "medusa_heads_topk", "medusa_heads_topk_workspace", "build_candidates", "tree_attention",
           "tree_attention_workspace", "evaluate_posterior", "evaluate_posterior_workspace", "kv_compact",
           "get_error", "fill_normal", "selftest_wait_timeout", "DTYPE_BF16", "DTYPE_F32", "MAX_NODES",
           "MAX_DEPTH", "EXPORTED_SYMBOLS"]

MAX_NODES = 256
NOALLOC_MAX_NODES = 64
MAX_DEPTH = 8
MASK_WORDS = 4
GREEDY, TYPICAL = 0, 1
DTYPE_BF16, DTYPE_F32 = 0, 1
ROOT_ARGMAX, ROOT_TYPICAL, ROOT_NUCLEUS = 0, 1, 2

_lib = None


class MVError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        name = _lib.mv_status_string(status).decode() if _lib is not None else str(status)
        super().__init__(f"{what}: {name} (status {status})")


class TreeDesc(ctypes.Structure):
    _fields_ = [("n_nodes", ctypes.c_int32), ("n_paths", ctypes.c_int32), ("depth", ctypes.c_int32),
                ("topk", ctypes.c_int32),
                ("tree_indices", ctypes.POINTER(ctypes.c_int32)), ("position_ids", ctypes.POINTER(ctypes.c_int32)),
                ("retrieve", ctypes.POINTER(ctypes.c_int32)), ("parent", ctypes.POINTER(ctypes.c_int32)),
                ("ancestors", ctypes.POINTER(ctypes.c_uint64)),
                ("d_tree_indices", ctypes.c_void_p), ("d_position_ids", ctypes.c_void_p),
                ("d_retrieve", ctypes.c_void_p), ("d_parent", ctypes.c_void_p), ("d_ancestors", ctypes.c_void_p)]


class AcceptParams(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int32), ("temperature", ctypes.c_float), ("eps", ctypes.c_float),
                ("delta", ctypes.c_float)]

    def __init__(self, mode=GREEDY, temperature=0.7, eps=0.09, delta=0.3):
        super().__init__(mode, temperature, eps, delta)


class RootParams(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int32), ("temperature", ctypes.c_float), ("eps", ctypes.c_float),
                ("delta", ctypes.c_float), ("top_p", ctypes.c_float), ("reserved", ctypes.c_uint32),
                ("key", ctypes.c_uint64)]

    def __init__(self, mode=ROOT_ARGMAX, temperature=0.7, eps=0.09, delta=0.3, top_p=0.8, key=0):
        super().__init__(mode, temperature, eps, delta, top_p, 0, key % 2 ** 64)


class PosteriorResult(ctypes.Structure):
    _fields_ = [("best", ctypes.c_int32), ("acc", ctypes.c_int32), ("next_node", ctypes.c_int32),
                ("next_root", ctypes.c_int32), ("n_tokens", ctypes.c_int32),
                ("nodes", ctypes.c_int32 * (MAX_DEPTH + 1)), ("tokens", ctypes.c_int32 * (MAX_DEPTH + 1))]


RESULT_INTS = ctypes.sizeof(PosteriorResult) // 4

_P, _I, _U, _F, _S = ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint32, ctypes.c_float, ctypes.c_size_t
_SIGS = {
    "mv_tree_create": ([_P, _P, _I, _I, ctypes.POINTER(_P)], _I),
    "mv_tree_describe": ([_P, ctypes.POINTER(TreeDesc)], _I),
    "mv_tree_destroy": ([_P], None),
    "medusa_heads_topk_workspace": ([_I, _I, _I, _I, _I, ctypes.POINTER(_S)], _I),
    "medusa_heads_topk": ([_P, _I, _I, _I, _P, _P, _I, _I, _P, _P, _P, _P, _P, _S, _P], _I),
    "build_candidates": ([_P, _P, _I, _I, _P, _P, _P, _P], _I),
    "tree_attention_workspace": ([_I, _I, _I, _I, ctypes.POINTER(_S)], _I),
    "tree_attention": ([_P, _P, _P, _I, _I, _I, _I, _P, _F, _P, _P, _S, _P], _I),
    "evaluate_posterior_workspace": ([_I, ctypes.POINTER(_S)], _I),
    "evaluate_posterior": ([_P, _I, _I, _P, _P, AcceptParams, _P, _P, _P, _P, _S, _P], _I),
    "kv_compact": ([_P, _I, _I, _I, _I, _I, _P, _P, _P], _I),
    "sample_root": ([_P, _I, RootParams, ctypes.c_uint64, _P, _P], _I),
    "evaluate_posterior_noalloc": ([_P, _I, _I, _P, _P, AcceptParams, _P, _P, _P, _P], _I),
    "mv_linear_bf16_workspace": ([ctypes.POINTER(_S)], _I),
    "mv_linear_bf16": ([_P, _P, _P, _I, _I, _I, _I, _P, _S, _P], _I),
    "mv_linear_bf16_packed": ([_P, _P, _P, _I, _I, _I, _I, _P, _S, _P], _I),
    "mv_packed_weight_bytes": ([_I, _I, _I, ctypes.POINTER(_S)], _I),
    "mv_pack_weight": ([_P, _P, _I, _I, _I, _P], _I),
    "mv_model_create": ([_P, _P, ctypes.POINTER(_P)], _I),
    "mv_model_create_f32": ([_P, _P, ctypes.POINTER(_P)], _I),
    "mv_model_create_random": ([_P, ctypes.c_uint64, ctypes.c_double, _I, ctypes.POINTER(_P)], _I),
    "mv_model_dtype": ([_P], _I),
    "mv_model_destroy": ([_P], None),
    "mv_fill_normal": ([_P, _I, ctypes.c_int64, ctypes.c_uint64, ctypes.c_char_p, ctypes.c_double, _P], _I),
    "mv_session_workspace": ([_P, _I, _I, ctypes.POINTER(_S)], _I),
    "mv_session_create": ([_P, _P, _P, _I, _I, _P, _S, ctypes.POINTER(_P)], _I),
    "mv_batch_session_create": ([_P, _P, _I, _P, _I, _I, _P, _S, ctypes.POINTER(_P)], _I),
    "mv_session_destroy": ([_P], None),
    "mv_session_state": ([_P, _P], _I),
    "mv_prefill": ([_P, _P, _I, _P], _I),
    "mv_prefill_seq": ([_P, _I, _P, _I, _P], _I),
    "mv_session_set_root_sampling": ([_P, RootParams, ctypes.c_uint64, _P], _I),
    "medusa_verify_step": ([_P, AcceptParams, _P], _I),
    "medusa_verify_step_host": ([_P, AcceptParams, _P, _P, _P, _P], _I),
    "medusa_verify_steps_graph": ([_P, AcceptParams, _I, _P], _I),
    "mv_session_profile": ([_P, _I], _I),
    "mv_session_profile_read": ([_P, _P, _P], _I),
    "mv_get_error": ([ctypes.POINTER(_U)], _I),
    "mv_get_error_detail": ([ctypes.POINTER(_U)], _I),
    "mv_selftest_wait_timeout": ([_U, _P, _P], _I),
    "mv_status_string": ([_I], ctypes.c_char_p),
}
EXPORTED_SYMBOLS = tuple(_SIGS)


def lib(auto_build: bool = True):
    """The loaded library (built first if missing or stale and ``auto_build``)."""
    global _lib
    if _lib is None:
        if auto_build:
            build()
        if not os.path.exists(LIB):
            raise RuntimeError(f"{LIB} is missing: build it with medusa_tree_speculative_verify_gb300.build.build()")
        L = ctypes.CDLL(LIB)
        for name, (args, res) in _SIGS.items():
            f = getattr(L, name)
            f.argtypes, f.restype = args, res
        _lib = L
    return _lib


def _check(status, what):
    if status != 0:
        raise MVError(status, what)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


class Tree:
    """A static token tree (owned library handle) built from rank tuples (root excluded)."""

    def __init__(self, choices, topk):
        L = lib()
        ranks = [int(r) for c in choices for r in c]
        lens = [len(c) for c in choices]
        ra = (ctypes.c_int32 * max(1, len(ranks)))(*ranks)
        la = (ctypes.c_int32 * max(1, len(lens)))(*lens)
        h = ctypes.c_void_p()
        _check(L.mv_tree_create(ra, la, len(lens), topk, ctypes.byref(h)), "mv_tree_create")
        self.handle = h
        d = TreeDesc()
        _check(L.mv_tree_describe(h, ctypes.byref(d)), "mv_tree_describe")
        self.n_nodes, self.n_paths, self.depth, self.topk = d.n_nodes, d.n_paths, d.depth, d.topk
        arr = lambda p, n: np.ctypeslib.as_array(p, shape=(n,)).copy()
        self.tree_indices = arr(d.tree_indices, self.n_nodes)
        self.position_ids = arr(d.position_ids, self.n_nodes)
        self.retrieve = arr(d.retrieve, self.n_paths * (self.depth + 1)).reshape(self.n_paths, self.depth + 1)
        self.parent = arr(d.parent, self.n_nodes)
        self.ancestors = arr(d.ancestors, self.n_nodes * MASK_WORDS).reshape(self.n_nodes, MASK_WORDS)
        self.d_ancestors = d.d_ancestors

    def attn_mask(self):
        n = self.n_nodes
        return np.array([[(int(self.ancestors[i, j >> 6]) >> (j & 63)) & 1 for j in range(n)] for i in range(n)],
                        dtype=np.uint8)

    def __del__(self):
        if getattr(self, "handle", None) is not None and _lib is not None:
            _lib.mv_tree_destroy(self.handle)
            self.handle = None


def _ws_size(fn, *args):
    n = ctypes.c_size_t()
    _check(fn(*args, ctypes.byref(n)), fn.__name__)
    return n.value


def medusa_heads_topk_workspace(B, d, K, V, topk):
    return _ws_size(lib().medusa_heads_topk_workspace, B, d, K, V, topk)


def medusa_heads_topk(h, w1, w2, topk, out_idx, out_val=None, w_lm=None, out_root=None, workspace=None,
                      stream=None):
    """h bf16 [B,d]; w1 bf16 [K,d,d]; w2 bf16 [K,V,d]; out_idx int32 [B,K,topk]; out_val fp32 [B,K,topk]."""
    B, d = h.shape
    K, V = w2.shape[0], w2.shape[1]
    _check(lib().medusa_heads_topk(_ptr(h), B, d, K, _ptr(w1), _ptr(w2), V, topk, _ptr(w_lm), _ptr(out_idx),
                                   _ptr(out_val), _ptr(out_root), _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), _stream(stream)),
           "medusa_heads_topk")


def build_candidates(root, head_topk, tree: Tree, tree_tokens, cart=None, stream=None):
    """root int32 [1]; head_topk int32 [K, ld]; tree_tokens int32 [n]; cart int32 [paths, depth+1]."""
    K, ld = head_topk.shape
    _check(lib().build_candidates(_ptr(root), _ptr(head_topk), K, ld, tree.handle, _ptr(tree_tokens), _ptr(cart),
                                  _stream(stream)), "build_candidates")


def tree_attention_workspace(H, D, S_max, n_nodes):
    return _ws_size(lib().tree_attention_workspace, H, D, S_max, n_nodes)


def tree_attention(q, k_cache, v_cache, prefix_len, tree: Tree, scale, out, workspace, stream=None):
    """q bf16 [n,H,D]; k_cache/v_cache bf16 [H,S_max,D]; out bf16 [n,H,D]."""
    H, S_max, D = k_cache.shape
    _check(lib().tree_attention(_ptr(q), _ptr(k_cache), _ptr(v_cache), H, D, S_max, prefix_len, tree.handle,
                                float(scale), _ptr(out), _ptr(workspace),
                                workspace.numel() * workspace.element_size(), _stream(stream)), "tree_attention")


def evaluate_posterior_workspace(n_nodes):
    return _ws_size(lib().evaluate_posterior_workspace, n_nodes)


def evaluate_posterior(logits, tree_tokens, tree: Tree, params: AcceptParams, out, workspace, node_stats=None,
                       node_argmax=None, stream=None):
    """logits fp32 [n, ld] (first V columns used, V = logits.shape[1] unless sliced); out int32 [RESULT_INTS]."""
    n, V = logits.shape
    ld = logits.stride(0)
    _check(lib().evaluate_posterior(_ptr(logits), V, ld, _ptr(tree_tokens), tree.handle, params, _ptr(out),
                                    _ptr(node_stats), _ptr(node_argmax), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(), _stream(stream)),
           "evaluate_posterior")


def evaluate_posterior_noalloc(logits, tree_tokens, tree: Tree, params: AcceptParams, out, node_stats=None,
                               node_argmax=None, stream=None):
    """evaluate_posterior with the library's fixed scratch array instead of a workspace (allocates nothing)."""
    n, V = logits.shape
    _check(lib().evaluate_posterior_noalloc(_ptr(logits), V, logits.stride(0), _ptr(tree_tokens), tree.handle,
                                            params, _ptr(out), _ptr(node_stats), _ptr(node_argmax), _stream(stream)),
           "evaluate_posterior_noalloc")


def kv_compact(kv, prefix_len, result, cur_len=None, stream=None):
    """kv bf16 [L,2,H,S_max,D]; result: the int32 posterior result buffer; cur_len int32 [1]."""
    L, two, H, S_max, D = kv.shape
    assert two == 2
    _check(lib().kv_compact(_ptr(kv), L, H, S_max, D, prefix_len, _ptr(result), _ptr(cur_len), _stream(stream)),
           "kv_compact")


def sample_root(logits_row, params: RootParams, counter, out, stream=None):
    """One root draw from logits_row fp32 [V] (contiguous) into out int32 [1] with generator counter ``counter``."""
    _check(lib().sample_root(_ptr(logits_row), logits_row.numel(), params, counter % 2 ** 64, _ptr(out),
                             _stream(stream)), "sample_root")


def get_error(with_detail=False):
    """(status, code[, detail]): reads and clears the device error word (synchronises the device)."""
    code, detail = ctypes.c_uint32(), ctypes.c_uint32()
    lib().mv_get_error_detail(ctypes.byref(detail))
    st = lib().mv_get_error(ctypes.byref(code))
    return (st, code.value, detail.value) if with_detail else (st, code.value)


def fill_normal(out, seed, name, std=1.0, stream=None):
    """Fills the contiguous bf16 or fp32 device tensor ``out`` with the library's N(0, std^2) stream ``name``
    under ``seed`` (see mv_fill_normal)."""
    import torch
    dt = DTYPE_F32 if out.dtype == torch.float32 else DTYPE_BF16
    assert out.dtype in (torch.float32, torch.bfloat16) and out.is_contiguous()
    _check(lib().mv_fill_normal(_ptr(out), dt, out.numel(), seed % 2 ** 64, name.encode(), float(std),
                                _stream(stream)), "mv_fill_normal")


def selftest_wait_timeout(limit_ns, out, stream=None):
    """Runs the library's two bounded waits on a counter and a barrier nothing completes (see
    mv_selftest_wait_timeout); out: int32 [4] device tensor."""
    _check(lib().mv_selftest_wait_timeout(limit_ns, _ptr(out), _stream(stream)), "mv_selftest_wait_timeout")


def result_dict(buf):
    """Decode a PosteriorResult from an int32 tensor / array of RESULT_INTS entries."""
    a = np.asarray(buf.cpu() if hasattr(buf, "cpu") else buf, dtype=np.int32)
    r = PosteriorResult.from_buffer_copy(a.tobytes())
    return dict(best=r.best, acc=r.acc, next_node=r.next_node, next_root=r.next_root, n_tokens=r.n_tokens,
                nodes=list(r.nodes)[: r.acc + 1], tokens=list(r.tokens)[: r.acc + 1])


# --------------------------------------------------------------------------------------------- projections

def linear_bf16_workspace():
    return _ws_size(lib().mv_linear_bf16_workspace)


def linear_bf16(w, x, out, workspace, stream=None):
    """out[:n, :M] (fp32) = x[n, K] @ w[M, K]^T on the tcgen05 kernel; out may have a row stride >= M."""
    M, K = w.shape
    n = x.shape[0]
    _check(lib().mv_linear_bf16(_ptr(w), _ptr(x), _ptr(out), M, K, n, out.stride(0), _ptr(workspace),
                                workspace.numel() * workspace.element_size(), _stream(stream)), "mv_linear_bf16")


def linear_bf16_packed(w_packed, M, K, x, out, workspace, stream=None):
    """linear_bf16 with the weight in the packed layout (pack_weight(w, 128))."""
    n = x.shape[0]
    _check(lib().mv_linear_bf16_packed(_ptr(w_packed), _ptr(x), _ptr(out), M, K, n, out.stride(0), _ptr(workspace),
                                       workspace.numel() * workspace.element_size(), _stream(stream)),
           "mv_linear_bf16_packed")


def pack_weight(w, tile_rows, stream=None, out=None):
    """w [M, K] in the projection kernel's packed layout (see mv_pack_weight), in a new bf16 tensor or in ``out``
    (a bf16 tensor of at least mv_packed_weight_bytes / 2 elements)."""
    import torch
    M, K = w.shape
    nbytes = _ws_size(lib().mv_packed_weight_bytes, M, K, tile_rows)
    if out is None:
        out = torch.empty(nbytes // 2, dtype=torch.bfloat16, device=w.device)
    elif out.dtype != torch.bfloat16 or out.numel() * 2 < nbytes:
        raise ValueError("pack_weight: out is not a bf16 tensor of the packed size")
    _check(lib().mv_pack_weight(_ptr(w), _ptr(out), M, K, tile_rows, _stream(stream)), "mv_pack_weight")
    return out


def pack_model_weights(w, drop_source=False):
    """Model weights with the projection matrices packed (embed and the Medusa matrices unchanged). A layer's
    gate and up matrices share one allocation, up right after gate, so the projection kernel loads the gate and
    up rows of a k-block with one copy."""
    import torch
    out = dict(w)
    for key, tr in (("wqkv", 128), ("wo", 128), ("w_down", 128)):
        packed = []
        for i in range(len(w[key])):
            packed.append(pack_weight(w[key][i], tr))
            if drop_source:
                w[key][i] = None
        out[key] = packed
    gates, ups = [], []
    for i in range(len(w["w_gate"])):
        F, K = w["w_gate"][i].shape
        n = _ws_size(lib().mv_packed_weight_bytes, F, K, 64) // 2
        both = torch.empty(2 * n, dtype=torch.bfloat16, device=w["w_gate"][i].device)
        gates.append(pack_weight(w["w_gate"][i], 64, out=both[:n]))
        ups.append(pack_weight(w["w_up"][i], 64, out=both[n:]))
        if drop_source:
            w["w_gate"][i] = None
            w["w_up"][i] = None
    out["w_gate"], out["w_up"] = gates, ups
    out["lm_head"] = pack_weight(w["lm_head"], 128)
    out["packed"] = True
    return out


# --------------------------------------------------------------------------------------------- model / session

class ModelDims(ctypes.Structure):
    _fields_ = [("d", _I), ("n_layers", _I), ("n_heads", _I), ("head_dim", _I), ("ffn", _I), ("vocab", _I),
                ("n_medusa", _I), ("rope_theta", _F), ("norm_eps", _F)]


class _Weights(ctypes.Structure):
    _fields_ = [("embed", _P), ("wqkv", _P), ("wo", _P), ("w_gate", _P), ("w_up", _P), ("w_down", _P),
                ("lm_head", _P), ("medusa_w1", _P), ("medusa_w2", _P), ("packed", _I)]


class _WeightsF32(ctypes.Structure):
    _fields_ = [("embed", _P), ("wqkv", _P), ("wo", _P), ("w_gate", _P), ("w_up", _P), ("w_down", _P),
                ("lm_head", _P), ("medusa_w1", _P), ("medusa_w2", _P)]


class _StatePtrs(ctypes.Structure):
    _fields_ = [("cur_len", _P), ("result", _P), ("head_topk", _P), ("tree_tokens", _P), ("cart", _P),
                ("logits", _P), ("ld_logits", _I), ("hidden", _P), ("root_counter", _P), ("batch", _I)]


def _c_dims(dims):
    return ModelDims(dims.d, dims.n_layers, dims.n_heads, dims.head_dim, dims.ffn, dims.vocab, dims.n_medusa,
                     dims.rope_theta, dims.norm_eps)


class Model:
    """A model handle over caller-owned device weights: bf16 (mv_model_create) or fp32 (mv_model_create_f32),
    chosen by the dtype of ``w["embed"]``.

    ``w`` maps embed, lm_head, medusa_w1 [K,d,d], medusa_w2 [K,V,d] to tensors and wqkv, wo, w_gate, w_up,
    w_down to per-layer lists of tensors (see mv_model_weights in include/medusa_verify.h). ``Model.random``
    makes a model whose weights the library draws and owns.
    """

    def __init__(self, dims, w):
        import torch
        self.dims = _c_dims(dims)
        self.w = w  # keep the tensors alive
        L = dims.n_layers
        arrs = {k: (ctypes.c_void_p * L)(*[t.data_ptr() for t in w[k]]) for k in
                ("wqkv", "wo", "w_gate", "w_up", "w_down")}
        self._arrs = arrs
        lists = [ctypes.cast(arrs[k], _P) for k in ("wqkv", "wo", "w_gate", "w_up", "w_down")]
        heads = (w["lm_head"].data_ptr(), w["medusa_w1"].data_ptr(), w["medusa_w2"].data_ptr())
        h = ctypes.c_void_p()
        if w["embed"].dtype == torch.float32:
            self.dtype = DTYPE_F32
            cw = _WeightsF32(w["embed"].data_ptr(), *lists, *heads)
            _check(lib().mv_model_create_f32(ctypes.byref(self.dims), ctypes.byref(cw), ctypes.byref(h)),
                   "mv_model_create_f32")
        else:
            self.dtype = DTYPE_BF16
            cw = _Weights(w["embed"].data_ptr(), *lists, *heads, 1 if w.get("packed") else 0)
            _check(lib().mv_model_create(ctypes.byref(self.dims), ctypes.byref(cw), ctypes.byref(h)),
                   "mv_model_create")
        self.handle = h

    @classmethod
    def random(cls, dims, seed=0, std=None, dtype=DTYPE_BF16):
        """A random-init model whose weights the library draws (mv_model_create_random) and owns."""
        self = cls.__new__(cls)
        self.dims = _c_dims(dims)
        self.w = None
        self.dtype = dtype
        h = ctypes.c_void_p()
        std = dims.std if std is None else std
        _check(lib().mv_model_create_random(ctypes.byref(self.dims), seed % 2 ** 64, float(std), dtype,
                                            ctypes.byref(h)), "mv_model_create_random")
        self.handle = h
        return self

    def __del__(self):
        if getattr(self, "handle", None) is not None and _lib is not None:
            _lib.mv_model_destroy(self.handle)
            self.handle = None


class Session:
    """A decode session: model + tree + KV cache + workspace (allocated here). batch > 1: that many sequences
    verified together (KV cache [batch,L,2,H,s_max,D]); the state views then have a leading batch dimension."""

    def __init__(self, model: Model, tree: Tree, s_max, topk=None, kv=None, batch=1):
        import torch
        d = model.dims
        self.model, self.tree, self.s_max, self.batch = model, tree, s_max, batch
        self.topk = topk or tree.topk
        shape = (d.n_layers, 2, d.n_heads, s_max, d.head_dim)
        if batch > 1:
            shape = (batch,) + shape
        kv_dtype = torch.float32 if getattr(model, "dtype", DTYPE_BF16) == DTYPE_F32 else torch.bfloat16
        self.kv = kv if kv is not None else torch.zeros(*shape, dtype=kv_dtype, device="cuda")
        nbytes = _ws_size(lib().mv_session_workspace, model.handle, s_max, self.topk)
        self.ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
        h = ctypes.c_void_p()
        _check(lib().mv_batch_session_create(model.handle, tree.handle, batch, _ptr(self.kv), s_max, self.topk,
                                             _ptr(self.ws), nbytes, ctypes.byref(h)), "mv_batch_session_create")
        self.handle = h
        sp = _StatePtrs()
        _check(lib().mv_session_state(h, ctypes.byref(sp)), "mv_session_state")
        base = self.ws.data_ptr()

        def view(ptr, count, dtype):
            off = ptr - base
            esz = torch.empty(0, dtype=dtype).element_size()
            return self.ws[off: off + count * esz].view(dtype)

        K, B = d.n_medusa, batch
        if B == 1:
            self.cur_len = view(sp.cur_len, 1, torch.int32)
            self.result = view(sp.result, RESULT_INTS, torch.int32)
            self.head_topk = view(sp.head_topk, K * self.topk, torch.int32).view(K, self.topk)
        else:
            self.cur_len = view(sp.cur_len, B, torch.int32)
            self.result = view(sp.result, B * RESULT_INTS, torch.int32).view(B, RESULT_INTS)
            self.head_topk = view(sp.head_topk, B * K * self.topk, torch.int32).view(B, K, self.topk)
        # the tree tokens of sequence b start at row 64 b (a batch of one: rows 0 .. n - 1)
        self.tree_tokens = view(sp.tree_tokens, tree.n_nodes if B == 1 else 64 * (B - 1) + tree.n_nodes,
                                torch.int32)
        self.cart = view(sp.cart, tree.n_paths * (tree.depth + 1), torch.int32).view(tree.n_paths, tree.depth + 1)
        self.ld_logits = sp.ld_logits
        self.logits = view(sp.logits, MAX_NODES * sp.ld_logits, torch.float32).view(MAX_NODES, sp.ld_logits)[:, : d.vocab]
        self.hidden = view(sp.hidden, MAX_NODES * d.d, torch.float32).view(MAX_NODES, d.d)
        self.root_counter = view(sp.root_counter, B, torch.int64)

    def prefill(self, tokens, stream=None):
        _check(lib().mv_prefill(self.handle, _ptr(tokens), tokens.numel(), _stream(stream)), "mv_prefill")

    def prefill_seq(self, seq, tokens, stream=None):
        _check(lib().mv_prefill_seq(self.handle, seq, _ptr(tokens), tokens.numel(), _stream(stream)), "mv_prefill_seq")

    def set_root_sampling(self, params: RootParams, counter=0, stream=None):
        """Draw the root after prefill / every step with ``params`` (ROOT_ARGMAX restores the argmax root)."""
        _check(lib().mv_session_set_root_sampling(self.handle, params, counter % 2 ** 64, _stream(stream)),
               "mv_session_set_root_sampling")

    def step(self, params: AcceptParams = None, stream=None):
        _check(lib().medusa_verify_step(self.handle, params or AcceptParams(), _stream(stream)), "medusa_verify_step")

    def steps_graph(self, n_steps, params: AcceptParams = None, stream=None):
        """n_steps verify steps replayed as one CUDA graph (captured on first use)."""
        _check(lib().medusa_verify_steps_graph(self.handle, params or AcceptParams(), n_steps, _stream(stream)),
               "medusa_verify_steps_graph")

    def step_host(self, params, seeds_in, result_out, seeds_out=None, stream=None):
        """Host-buffer step: seeds_in/out int32 [1 + K*topk] (pinned CPU tensors or None), result_out int32."""
        _check(lib().medusa_verify_step_host(self.handle, params, _ptr(seeds_in), _ptr(result_out), _ptr(seeds_out),
                                             _stream(stream)), "medusa_verify_step_host")

    def read_result(self, seq=None):
        """The last verification of the session (batch 1) or of sequence ``seq``."""
        return result_dict(self.result if seq is None and self.batch == 1 else self.result[seq or 0])

    def __del__(self):
        if getattr(self, "handle", None) is not None and _lib is not None:
            _lib.mv_session_destroy(self.handle)
            self.handle = None


PROF_KINDS = ("gemm_qkv", "attention", "gemm_o", "gemm_gate_up", "gemm_down", "gemm_lm", "posterior", "kv_compact",
              "heads", "other", "gemm_chain")


class Profiler:
    """Per-kind summed kernel milliseconds of a session (CUDA events around every launch)."""

    def __init__(self, sess: Session):
        self.sess = sess

    def enable(self):
        _check(lib().mv_session_profile(self.sess.handle, 1), "mv_session_profile")

    def disable(self):
        _check(lib().mv_session_profile(self.sess.handle, 0), "mv_session_profile")

    def read(self):
        ms = (ctypes.c_float * len(PROF_KINDS))()
        cnt = (ctypes.c_int32 * len(PROF_KINDS))()
        _check(lib().mv_session_profile_read(self.sess.handle, ms, cnt), "mv_session_profile_read")
        return {k: (float(ms[i]), int(cnt[i])) for i, k in enumerate(PROF_KINDS)}
