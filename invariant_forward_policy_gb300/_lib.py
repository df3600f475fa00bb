"""Thin ctypes binding of libbi.so: the same entry points as include/bi.h.

Every function takes torch tensors (or raw integer device addresses, or None
for NULL), passes their device pointers and the current CUDA stream to the C
ABI, and raises BiError on a non-zero status.  No arithmetic happens here.
If the library has not been built, loading fails loudly: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

BI_OK = 0
BI_ERR_INVALID_ARG = 1
BI_ERR_UNSUPPORTED_SHAPE = 2
BI_ERR_CUDA = 3
BI_ERR_DEVICE_CHECK = 4
BI_ERR_TIMEOUT = 5
BI_INVARIANT = 0
BI_FAST = 1
BI_DTYPE_BF16 = 0
BI_DTYPE_FP32 = 1
BI_EPI_NONE = 0
BI_EPI_SWIGLU = 1

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libbi.so")

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_int = ctypes.c_int
_f32 = ctypes.c_float
_f64 = ctypes.c_double
_sz = ctypes.c_size_t


class BiError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"bi status {status}: {msg}")
        self.status = status


class bi_model_config(ctypes.Structure):
    _fields_ = [("n_layers", _i64), ("d", _i64), ("n_heads_q", _i64), ("n_heads_kv", _i64), ("head_dim", _i64),
                ("ffn", _i64), ("vocab", _i64), ("eps", _f32), ("rope_theta", _f32), ("kv_block", _i64),
                ("kv_split", _i64), ("max_pos", _i64), ("fp8", _i64)]


class bi_layer_weights(ctypes.Structure):
    _fields_ = [("attn_norm", _vp), ("wqkv", _vp), ("wo", _vp), ("ffn_norm", _vp), ("w13", _vp), ("w2", _vp),
                ("wqkv8", _vp), ("wqkv_s", _vp), ("wo8", _vp), ("wo_s", _vp), ("w138", _vp), ("w13_s", _vp),
                ("w28", _vp), ("w2_s", _vp)]


class bi_weights(ctypes.Structure):
    _fields_ = [("embed", _vp), ("final_norm", _vp), ("lm_head", _vp), ("layers", ctypes.POINTER(bi_layer_weights)),
                ("rope_table", _vp)]


_SIGS = {
    "bi_version": (_int, []),
    "bi_last_error": (ctypes.c_char_p, []),
    "bi_launch_count": (_i64, []),
    "bi_device_status": (_int, []),
    "bi_rmsnorm": (_int, [_vp, _vp, _vp, _vp, _i64, _i64, _f32, _int, _vp]),
    "bi_gemm": (_int, [_vp, _i64, _i64, _vp, _i64, _vp, _int, _int, _int, _vp, _sz, _vp]),
    "bi_gemm_workspace_size": (_sz, [_i64, _i64, _i64, _int, _int]),
    "bi_gemm_tile_n": (_int, [_i64, _i64, _int]),
    "bi_grouped_gemm": (_int, [_vp, _i64, _i64, _vp, _i64, _i64, _vp, _vp, _int, _int, _vp]),
    "bi_rope_kv_write": (_int, [_vp, _i64, _vp, _vp, _vp, _i64, _i64, _int, _int, _int, _vp, _i64, _vp, _i64, _i64,
                                _vp, _vp, _vp, _vp]),
    "bi_rope_table": (_int, [_vp, _i64, _int, _f64, _vp]),
    "bi_qkv_rope_kv_write": (_int, [_vp, _i64, _i64, _vp, _int, _int, _int, _vp, _vp, _vp, _i64, _vp, _i64, _i64, _vp,
                                    _vp, _vp, _int, _vp]),
    "bi_attention": (_int, [_vp, _i64, _vp, _vp, _vp, _i64, _i64, _int, _int, _int, _vp, _vp, _vp, _i64, _i64, _i64,
                            _int, _f32, _vp, _sz, _vp, _int, _vp]),
    "bi_attention_workspace_size": (_sz, [_i64, _int, _int, _i64, _int]),
    "bi_attention_static_scratch": (_int, [_vp, _i64, _vp, _vp, _vp, _i64, _i64, _int, _int, _int, _vp, _vp, _vp,
                                           _i64, _i64, _i64, _int, _f32, _vp, _int, _vp]),
    "bi_topk": (_int, [_vp, _i64, _i64, _vp, _int, _vp, _int, _vp]),
    "bi_quantize_fp8": (_int, [_vp, _i64, _i64, _int, _vp, _vp, _vp]),
    "bi_ssd_state_bytes": (_sz, [_int, _int, _int, _int, _int]),
    "bi_kv_fp8_write": (_int, [_vp, _vp, _i64, _vp, _vp, _vp, _i64, _i64, _int, _int, _vp, _i64, _i64, _vp, _vp, _vp,
                               _vp, _vp]),
    "bi_kv_fp8_gather": (_int, [_vp, _vp, _vp, _vp, _i64, _vp, _vp, _vp, _i64, _int, _int, _vp, _i64, _vp, _vp, _vp,
                                _vp]),
    "bi_attention_fp8": (_int, [_vp, _i64, _vp, _vp, _vp, _i64, _i64, _int, _int, _int, _vp, _vp, _vp, _vp, _vp,
                                _i64, _i64, _i64, _int, _f32, _vp, _sz, _vp, _vp, _vp, _int, _vp]),
    "bi_ssd_chunk_scan": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _int, _int, _int, _int, _int, _vp,
                                 _i64, _vp, _int, _vp]),
    "bi_gemm_fp8": (_int, [_vp, _vp, _i64, _i64, _vp, _vp, _i64, _vp, _int, _int, _vp]),
    "bi_rmsnorm_fp8": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _f32, _vp]),
    "bi_swiglu_fp8": (_int, [_vp, _i64, _i64, _vp, _vp, _vp]),
    "bi_embed": (_int, [_vp, _i64, _vp, _i64, _i64, _vp, _vp]),
    "bi_logprob_gather": (_int, [_vp, _vp, _i64, _i64, _vp, _vp, _int, _vp, _sz, _vp]),
    "bi_logprob_workspace_size": (_sz, [_i64, _i64, _int]),
    "bi_lm_head_logprob": (_int, [_vp, _i64, _i64, _vp, _i64, _vp, _vp, _vp, _int, _vp, _sz, _vp]),
    "bi_lm_head_logprob_workspace_size": (_sz, [_i64, _i64, _i64, _int]),
    "bi_moe_route_topk": (_int, [_vp, _i64, _int, _int, _vp, _vp, _vp]),
    "bi_moe_permute": (_int, [_vp, _i64, _int, _int, _i64, _vp, _vp, _vp, _vp, _sz, _vp]),
    "bi_moe_permute_workspace_size": (_sz, [_i64, _int, _int]),
    "bi_moe_permute_masked": (_int, [_vp, _i64, _int, _int, _i64, _vp, _vp, _vp, _sz, _vp]),
    "bi_moe_gather": (_int, [_vp, _vp, _i64, _int, _i64, _vp, _vp]),
    "bi_moe_combine": (_int, [_vp, _vp, _vp, _i64, _int, _i64, _vp, _int, _vp, _sz, _vp]),
    "bi_moe_combine_workspace_size": (_sz, [_i64, _i64, _int]),
    "bi_moe_layer": (_int, [_vp, _vp, _i64, _i64, _int, _int, _i64, _vp, _vp, _vp, _int, _vp, _sz, _vp]),
    "bi_moe_layer_workspace_size": (_sz, [_i64, _i64, _int, _int, _i64, _int]),
    "bi_model_create": (_int, [ctypes.POINTER(bi_model_config), ctypes.POINTER(bi_weights), _vp,
                               ctypes.POINTER(_vp)]),
    "bi_model_destroy": (None, [_vp]),
    "bi_model_set_dump": (_int, [_vp, _vp, _i64]),
    "bi_kv_cache_bytes": (_sz, [ctypes.POINTER(bi_model_config), _i64]),
    "bi_forward_workspace_size": (_sz, [ctypes.POINTER(bi_model_config), _i64, _i64, _i64, _i64, _int]),
    "bi_forward_prefill": (_int, [_vp, _vp, _vp, ctypes.POINTER(_i64), ctypes.POINTER(_i64), ctypes.POINTER(_i64),
                                  _i64, _i64, _vp, _i64, _vp, _vp, _i64, _vp, _vp, _vp, _sz, _i64, _i64, _i64, _int,
                                  _vp]),
    "bi_prefill_plan": (_i64, [ctypes.POINTER(_i64), ctypes.POINTER(_i64), ctypes.POINTER(_i64), _i64, _i64, _i64,
                               ctypes.POINTER(_i64), _i64]),
    "bi_forward_decode": (_int, [_vp, _vp, _vp, _i64, _vp, _i64, _vp, _vp, _i64, _i64, _vp, _vp, _vp, _sz, _int,
                                 _vp]),
    "bi_decode_advance": (_int, [_vp, _vp, _vp, _vp, _i64, _vp, _vp, _vp, _i64, _vp]),
}

EXPORTED = tuple(_SIGS)

_L = None


def load() -> ctypes.CDLL:
    """Load libbi.so (once).  Raises if it has not been built."""
    global _L
    if _L is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                               "(there is no CPU fallback)")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _L = lib
    return _L


def _p(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if isinstance(t, torch.Tensor):
        if t.numel() and not t.is_cuda:
            raise ValueError("tensor must live on the GPU")
        return t.data_ptr() if t.numel() else None
    raise TypeError(type(t))


def _s(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check(st: int):
    if st != BI_OK:
        raise BiError(st, load().bi_last_error().decode())


def _nb(t) -> int:
    return 0 if t is None else t.numel() * t.element_size()


# ---------------------------------------------------------------- entry points
def bi_version() -> int:
    return load().bi_version()


def bi_last_error() -> str:
    return load().bi_last_error().decode()


def bi_launch_count() -> int:
    return load().bi_launch_count()


def bi_device_status() -> int:
    return load().bi_device_status()


def bi_rmsnorm(x, residual, gamma, y, rows, d, eps=1e-6, mode=BI_INVARIANT, stream=None):
    _check(load().bi_rmsnorm(_p(x), _p(residual), _p(gamma), _p(y), rows, d, eps, mode, _s(stream)))


def bi_gemm(A, M, K, W, N, C, c_dtype=BI_DTYPE_BF16, epilogue=BI_EPI_NONE, mode=BI_INVARIANT, workspace=None,
            stream=None):
    _check(load().bi_gemm(_p(A), M, K, _p(W), N, _p(C), c_dtype, epilogue, mode, _p(workspace), _nb(workspace),
                          _s(stream)))


def bi_gemm_workspace_size(M, N, K, epilogue=BI_EPI_NONE, mode=BI_INVARIANT) -> int:
    return load().bi_gemm_workspace_size(M, N, K, epilogue, mode)


def bi_gemm_tile_n(N, K, epilogue=BI_EPI_NONE) -> int:
    return load().bi_gemm_tile_n(N, K, epilogue)


def bi_grouped_gemm(A, M_rows, K, W, E, N, tile_expert, C, c_dtype=BI_DTYPE_BF16, epilogue=BI_EPI_NONE, stream=None):
    _check(load().bi_grouped_gemm(_p(A), M_rows, K, _p(W), E, N, _p(tile_expert), _p(C), c_dtype, epilogue,
                                  _s(stream)))


def bi_qkv_rope_kv_write(x, T, K, wqkv, Hq, Hkv, hd, row_seq, row_pos, rope_table, max_pos, block_table,
                         max_blocks_per_seq, n_blocks, q_out, k_cache, v_cache, mode=BI_INVARIANT, stream=None):
    _check(load().bi_qkv_rope_kv_write(_p(x), T, K, _p(wqkv), Hq, Hkv, hd, _p(row_seq), _p(row_pos), _p(rope_table),
                                       max_pos, _p(block_table), max_blocks_per_seq, n_blocks, _p(q_out), _p(k_cache),
                                       _p(v_cache), mode, _s(stream)))


def bi_rope_table(table, max_pos, hd, theta=10000.0, stream=None):
    _check(load().bi_rope_table(_p(table), max_pos, hd, theta, _s(stream)))


def bi_rope_kv_write(qkv, T, piece_seq, piece_row0, piece_pos0, P, max_q_len, Hq, Hkv, hd, rope_table, max_pos,
                     block_table, max_blocks_per_seq, n_blocks, q_out, k_cache, v_cache, stream=None):
    _check(load().bi_rope_kv_write(_p(qkv), T, _p(piece_seq), _p(piece_row0), _p(piece_pos0), P, max_q_len, Hq, Hkv,
                                   hd, _p(rope_table), max_pos, _p(block_table), max_blocks_per_seq, n_blocks,
                                   _p(q_out), _p(k_cache), _p(v_cache), _s(stream)))


def bi_attention(q, T, piece_seq, piece_row0, piece_pos0, P, max_q_len, Hq, Hkv, hd, k_cache, v_cache, block_table,
                 max_blocks_per_seq, n_blocks, max_ctx, kv_split, scale, workspace, out, mode=BI_INVARIANT,
                 stream=None):
    _check(load().bi_attention(_p(q), T, _p(piece_seq), _p(piece_row0), _p(piece_pos0), P, max_q_len, Hq, Hkv, hd,
                               _p(k_cache), _p(v_cache), _p(block_table), max_blocks_per_seq, n_blocks, max_ctx,
                               kv_split, scale, _p(workspace), _nb(workspace), _p(out), mode, _s(stream)))


def bi_attention_fp8(q, T, piece_seq, piece_row0, piece_pos0, P, max_q_len, Hq, Hkv, hd, k_cache8, v_cache8, k_scale,
                     v_scale, block_table, max_blocks_per_seq, n_blocks, max_ctx, kv_split, scale, workspace, out,
                     out_q=None, out_scale=None, mode=BI_INVARIANT, stream=None):
    _check(load().bi_attention_fp8(_p(q), T, _p(piece_seq), _p(piece_row0), _p(piece_pos0), P, max_q_len, Hq, Hkv,
                                   hd, _p(k_cache8), _p(v_cache8), _p(k_scale), _p(v_scale), _p(block_table),
                                   max_blocks_per_seq, n_blocks, max_ctx, kv_split, scale, _p(workspace),
                                   _nb(workspace), _p(out), _p(out_q), _p(out_scale), mode, _s(stream)))


def bi_attention_static_scratch(q, T, piece_seq, piece_row0, piece_pos0, P, max_q_len, Hq, Hkv, hd, k_cache, v_cache,
                                block_table, max_blocks_per_seq, n_blocks, max_ctx, kv_split, scale, out,
                                mode=BI_INVARIANT, stream=None):
    """bi_attention without a caller workspace (the library's own static scratch array)."""
    _check(load().bi_attention_static_scratch(_p(q), T, _p(piece_seq), _p(piece_row0), _p(piece_pos0), P, max_q_len,
                                              Hq, Hkv, hd, _p(k_cache), _p(v_cache), _p(block_table),
                                              max_blocks_per_seq, n_blocks, max_ctx, kv_split, scale, _p(out), mode,
                                              _s(stream)))


def bi_attention_workspace_size(max_T, Hq, hd, max_ctx, kv_split) -> int:
    return load().bi_attention_workspace_size(max_T, Hq, hd, max_ctx, kv_split)


def bi_kv_fp8_write(k, v, T, piece_seq, piece_row0, piece_pos0, P, max_q_len, Hkv, hd, block_table,
                    max_blocks_per_seq, n_blocks, k_cache8, v_cache8, k_scale, v_scale, stream=None):
    _check(load().bi_kv_fp8_write(_p(k), _p(v), T, _p(piece_seq), _p(piece_row0), _p(piece_pos0), P, max_q_len, Hkv,
                                  hd, _p(block_table), max_blocks_per_seq, n_blocks, _p(k_cache8), _p(v_cache8),
                                  _p(k_scale), _p(v_scale), _s(stream)))


def bi_kv_fp8_gather(k_cache8, v_cache8, k_scale, v_scale, n_blocks, piece_seq, piece_row0, piece_pos0, P, Hkv, hd,
                     block_table, max_blocks_per_seq, k_ws, v_ws, ws_block_table, stream=None):
    _check(load().bi_kv_fp8_gather(_p(k_cache8), _p(v_cache8), _p(k_scale), _p(v_scale), n_blocks, _p(piece_seq),
                                   _p(piece_row0), _p(piece_pos0), P, Hkv, hd, _p(block_table), max_blocks_per_seq,
                                   _p(k_ws), _p(v_ws), _p(ws_block_table), _s(stream)))


def bi_ssd_state_bytes(H, G, P, N, Q) -> int:
    return load().bi_ssd_state_bytes(H, G, P, N, Q)


def bi_ssd_chunk_scan(x, B, C, loga, piece_seq, piece_row0, piece_pos0, pieces, max_q_len, H, G, P, N, Q, state, n_seq,
                      y, mode=BI_INVARIANT, stream=None):
    _check(load().bi_ssd_chunk_scan(_p(x), _p(B), _p(C), _p(loga), _p(piece_seq), _p(piece_row0), _p(piece_pos0),
                                    pieces, max_q_len, H, G, P, N, Q, _p(state), n_seq, _p(y), mode, _s(stream)))


def bi_quantize_fp8(x, R, C, block_rows, q, scales, stream=None):
    _check(load().bi_quantize_fp8(_p(x), R, C, block_rows, _p(q), _p(scales), _s(stream)))


def bi_gemm_fp8(Aq, sa, M, K, Wq, sw, N, C, c_dtype=BI_DTYPE_BF16, mode=BI_INVARIANT, stream=None):
    _check(load().bi_gemm_fp8(_p(Aq), _p(sa), M, K, _p(Wq), _p(sw), N, _p(C), c_dtype, mode, _s(stream)))


def bi_rmsnorm_fp8(x, residual, gamma, y, q, q_scale, rows, d, eps=1e-6, stream=None):
    _check(load().bi_rmsnorm_fp8(_p(x), _p(residual), _p(gamma), _p(y), _p(q), _p(q_scale), rows, d, eps,
                                 _s(stream)))


def bi_swiglu_fp8(g13, T, F, q, q_scale, stream=None):
    _check(load().bi_swiglu_fp8(_p(g13), T, F, _p(q), _p(q_scale), _s(stream)))


def bi_topk(scores, T, ld, n_valid, K, idx_out, mode=BI_INVARIANT, stream=None):
    _check(load().bi_topk(_p(scores), T, ld, _p(n_valid), K, _p(idx_out), mode, _s(stream)))


def bi_embed(ids, T, table, V, d, out, stream=None):
    _check(load().bi_embed(_p(ids), T, _p(table), V, d, _p(out), _s(stream)))


def bi_logprob_gather(logits, ids, T, V, logprob_out, argmax_out=None, mode=BI_INVARIANT, workspace=None,
                      stream=None):
    _check(load().bi_logprob_gather(_p(logits), _p(ids), T, V, _p(logprob_out), _p(argmax_out), mode, _p(workspace),
                                    _nb(workspace), _s(stream)))


def bi_logprob_workspace_size(T, V, mode=BI_INVARIANT) -> int:
    return load().bi_logprob_workspace_size(T, V, mode)


def bi_lm_head_logprob(X, T, K, W, V, ids, logprob_out, argmax_out=None, mode=BI_INVARIANT, workspace=None,
                       stream=None):
    _check(load().bi_lm_head_logprob(_p(X), T, K, _p(W), V, _p(ids), _p(logprob_out), _p(argmax_out), mode,
                                     _p(workspace), _nb(workspace), _s(stream)))


def bi_lm_head_logprob_workspace_size(T, V, K, mode=BI_INVARIANT) -> int:
    return load().bi_lm_head_logprob_workspace_size(T, V, K, mode)


def bi_moe_route_topk(logits, T, E, k, ids, weights, stream=None):
    _check(load().bi_moe_route_topk(_p(logits), T, E, k, _p(ids), _p(weights), _s(stream)))


def bi_moe_permute(ids, T, k, E, max_rows, row_of_slot, tile_expert, expert_offsets, workspace, stream=None):
    _check(load().bi_moe_permute(_p(ids), T, k, E, max_rows, _p(row_of_slot), _p(tile_expert), _p(expert_offsets),
                                 _p(workspace), _nb(workspace), _s(stream)))


def bi_moe_permute_workspace_size(T, k, E) -> int:
    return load().bi_moe_permute_workspace_size(T, k, E)


def bi_moe_permute_masked(ids, T, k, E, capacity, row_of_slot, tile_expert, workspace, stream=None):
    _check(load().bi_moe_permute_masked(_p(ids), T, k, E, capacity, _p(row_of_slot), _p(tile_expert), _p(workspace),
                                        _nb(workspace), _s(stream)))


def bi_moe_gather(x, row_of_slot, T, k, d, xp, stream=None):
    _check(load().bi_moe_gather(_p(x), _p(row_of_slot), T, k, d, _p(xp), _s(stream)))


def bi_moe_combine(y, row_of_slot, w, T, k, d, out, mode=BI_INVARIANT, workspace=None, stream=None):
    _check(load().bi_moe_combine(_p(y), _p(row_of_slot), _p(w), T, k, d, _p(out), mode, _p(workspace), _nb(workspace),
                                 _s(stream)))


def bi_moe_combine_workspace_size(T, d, mode=BI_INVARIANT) -> int:
    return load().bi_moe_combine_workspace_size(T, d, mode)


def bi_moe_layer(x, router_logits, T, d, E, k, F, w13, w2, out, mode=BI_INVARIANT, workspace=None, stream=None):
    _check(load().bi_moe_layer(_p(x), _p(router_logits), T, d, E, k, F, _p(w13), _p(w2), _p(out), mode,
                               _p(workspace), _nb(workspace), _s(stream)))


def bi_moe_layer_workspace_size(T, d, E, k, F, mode=BI_INVARIANT) -> int:
    return load().bi_moe_layer_workspace_size(T, d, E, k, F, mode)


def bi_model_create(cfg: bi_model_config, weights: bi_weights, stream=None) -> int:
    h = _vp()
    _check(load().bi_model_create(ctypes.byref(cfg), ctypes.byref(weights), _s(stream), ctypes.byref(h)))
    return h.value


def bi_model_destroy(handle: int):
    load().bi_model_destroy(handle)


def bi_model_set_dump(handle: int, dump, max_rows: int):
    _check(load().bi_model_set_dump(handle, _p(dump), max_rows))


def bi_kv_cache_bytes(cfg: bi_model_config, n_blocks: int) -> int:
    return load().bi_kv_cache_bytes(ctypes.byref(cfg), n_blocks)


def bi_forward_workspace_size(cfg: bi_model_config, max_tokens, max_pieces, max_ctx, max_logit_rows,
                              mode=BI_INVARIANT) -> int:
    return load().bi_forward_workspace_size(ctypes.byref(cfg), max_tokens, max_pieces, max_ctx, max_logit_rows, mode)


def _i64_array(vals):
    if vals is None:
        return None
    arr = (_i64 * len(vals))(*[int(v) for v in vals])
    return arr


def bi_forward_prefill(model, tokens, target_ids, cu_seqlens, start_pos, logit_from, B, chunk, block_table,
                       max_blocks_per_seq, k_cache, v_cache, n_blocks, logprob_out, sampled_out, workspace, max_tokens,
                       max_ctx, max_logit_rows, mode=BI_INVARIANT, stream=None):
    cu = _i64_array(cu_seqlens)
    sp = _i64_array(start_pos)
    lf = _i64_array(logit_from)
    _check(load().bi_forward_prefill(model, _p(tokens), _p(target_ids), cu, sp, lf, B, chunk, _p(block_table),
                                     max_blocks_per_seq, _p(k_cache), _p(v_cache), n_blocks, _p(logprob_out),
                                     _p(sampled_out), _p(workspace), _nb(workspace), max_tokens, max_ctx,
                                     max_logit_rows, mode, _s(stream)))


def bi_prefill_plan(cu_seqlens, start_pos, logit_from, chunk, max_tokens):
    """The pass schedule bi_forward_prefill runs (host only): a list of records
    (pass, seq, row0, rows, pos0, tok0, lfirst, loff), one per piece, in launch order."""
    B = len(cu_seqlens) - 1
    cu, sp, lf = _i64_array(cu_seqlens), _i64_array(start_pos), _i64_array(logit_from)
    n = load().bi_prefill_plan(cu, sp, lf, B, chunk, max_tokens, None, 0)
    if n < 0:
        raise BiError(BI_ERR_INVALID_ARG, "bi_prefill_plan: invalid arguments")
    out = (_i64 * (8 * max(n, 1)))()
    load().bi_prefill_plan(cu, sp, lf, B, chunk, max_tokens, out, n)
    return [tuple(out[8 * r: 8 * r + 8]) for r in range(n)]


def bi_forward_decode(model, tokens, pos, B, block_table, max_blocks_per_seq, k_cache, v_cache, n_blocks, max_ctx,
                      sampled_out, logprob_out, workspace, mode=BI_INVARIANT, stream=None):
    _check(load().bi_forward_decode(model, _p(tokens), _p(pos), B, _p(block_table), max_blocks_per_seq, _p(k_cache),
                                    _p(v_cache), n_blocks, max_ctx, _p(sampled_out), _p(logprob_out), _p(workspace),
                                    _nb(workspace), mode, _s(stream)))


def bi_decode_advance(sampled, logprob, tokens, pos, B, step_counter, hist_ids, hist_lp, max_steps, stream=None):
    _check(load().bi_decode_advance(_p(sampled), _p(logprob), _p(tokens), _p(pos), B, _p(step_counter), _p(hist_ids),
                                    _p(hist_lp), max_steps, _s(stream)))
