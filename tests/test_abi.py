"""The C-ABI library loads, exports every symbol its header declares, and
rejects bad arguments before launching anything (no GPU needed)."""
import ctypes
import os
import re

import pytest

import invariant_forward_policy_gb300 as bi
from invariant_forward_policy_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "bi.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(bi_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    return _lib.load()


def test_every_declared_symbol_is_exported_and_bound(lib):
    names = _declared()
    assert len(names) >= 30
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(_lib.EXPORTED) == names


def test_version_and_no_error(lib):
    assert bi.bi_version() == 100
    assert isinstance(bi.bi_last_error(), str)


def test_validation_rejects_bad_arguments_without_launching(lib):
    # null pointers, bad shapes and bad modes are refused before any CUDA call
    assert lib.bi_rmsnorm(None, None, None, None, 4, 64, 1e-6, 0, None) == bi.BI_ERR_INVALID_ARG
    assert "null" in bi.bi_last_error()
    assert lib.bi_rmsnorm(16, None, 16, 16, 4, 63, 1e-6, 0, None) == bi.BI_ERR_INVALID_ARG
    assert lib.bi_rmsnorm(16, None, 16, 16, 4, 64, 1e-6, 7, None) == bi.BI_ERR_INVALID_ARG
    assert lib.bi_gemm(16, 4, 100, 16, 64, 16, 0, 0, 0, None, 0, None) == bi.BI_ERR_UNSUPPORTED_SHAPE
    assert lib.bi_gemm(16, 4, 64, 16, 64, 16, 0, 5, 0, None, 0, None) == bi.BI_ERR_INVALID_ARG
    assert lib.bi_gemm(17, 4, 64, 16, 64, 16, 0, 0, 0, None, 0, None) == bi.BI_ERR_INVALID_ARG  # misaligned
    assert lib.bi_logprob_gather(16, None, 4, 6, 16, None, 0, None, 0, None) == bi.BI_ERR_INVALID_ARG
    assert lib.bi_moe_route_topk(16, 4, 65, 8, 16, 16, None) == bi.BI_ERR_UNSUPPORTED_SHAPE
    assert lib.bi_moe_route_topk(16, 4, 64, 65, 16, 16, None) == bi.BI_ERR_INVALID_ARG
    assert lib.bi_attention(16, 4, 16, 16, 16, 1, 4, 8, 8, 96, 16, 16, 16, 1, 1, 64, 512, 0.1, 16, 1 << 20, 16, 0,
                            None) == bi.BI_ERR_UNSUPPORTED_SHAPE
    assert lib.bi_attention(16, 4, 16, 16, 16, 1, 4, 8, 8, 64, 16, 16, 16, 1, 1, 64, 500, 0.1, 16, 1 << 20, 16, 0,
                            None) == bi.BI_ERR_INVALID_ARG
    assert lib.bi_quantize_fp8(16, 4, 100, 1, 16, 16, None) == bi.BI_ERR_UNSUPPORTED_SHAPE   # C % 128
    assert lib.bi_quantize_fp8(16, 4, 128, 64, 16, 16, None) == bi.BI_ERR_INVALID_ARG        # block rows
    assert lib.bi_gemm_fp8(16, 16, 4, 100, 16, 16, 128, 16, 0, 0, None) == bi.BI_ERR_UNSUPPORTED_SHAPE
    assert lib.bi_gemm_fp8(16, 16, 4, 128, 16, 16, 128, 16, 7, 0, None) == bi.BI_ERR_INVALID_ARG
    assert lib.bi_rmsnorm_fp8(16, None, 16, None, 16, 16, 4, 200, 1e-6, None) == bi.BI_ERR_UNSUPPORTED_SHAPE
    assert lib.bi_rmsnorm_fp8(16, None, 16, None, None, 16, 4, 256, 1e-6, None) == bi.BI_ERR_INVALID_ARG
    assert lib.bi_swiglu_fp8(16, 4, 200, 16, 16, None) == bi.BI_ERR_INVALID_ARG
    # FP8 attention: scales missing; quantised output needs Hq*hd % 128 == 0 and both of out_q / out_scale
    assert lib.bi_attention_fp8(16, 4, 16, 16, 16, 1, 4, 8, 8, 64, 16, 16, None, 16, 16, 1, 1, 64, 512, 0.1, 16,
                                1 << 20, 16, None, None, 0, None) == bi.BI_ERR_INVALID_ARG
    assert lib.bi_attention_fp8(16, 4, 16, 16, 16, 1, 4, 1, 1, 64, 16, 16, 16, 16, 16, 1, 1, 64, 512, 0.1, 16,
                                1 << 20, None, 16, 16, 0, None) == bi.BI_ERR_UNSUPPORTED_SHAPE
    assert lib.bi_attention_fp8(16, 4, 16, 16, 16, 1, 4, 8, 8, 64, 16, 16, 16, 16, 16, 1, 1, 64, 512, 0.1, 16,
                                1 << 20, 16, 16, None, 0, None) == bi.BI_ERR_INVALID_ARG
    assert lib.bi_topk(16, 4, 64, 16, 0, 16, 0, None) == bi.BI_ERR_INVALID_ARG       # K < 1
    assert lib.bi_topk(16, 4, 64, 16, 4097, 16, 0, None) == bi.BI_ERR_INVALID_ARG    # K > 4096
    assert lib.bi_topk(None, 4, 64, 16, 8, 16, 0, None) == bi.BI_ERR_INVALID_ARG     # null scores
    assert lib.bi_topk(16, 4, 64, 16, 8, 16, 3, None) == bi.BI_ERR_INVALID_ARG       # bad mode
    # empty inputs are no-ops
    assert lib.bi_rmsnorm(None, None, None, None, 0, 64, 1e-6, 0, None) == bi.BI_OK
    assert lib.bi_topk(None, 0, 64, None, 8, None, 0, None) == bi.BI_OK
    assert lib.bi_gemm(None, 0, 64, None, 64, None, 0, 0, 0, None, 0, None) == bi.BI_OK


def test_model_config_validation(lib):
    cfg = _lib.bi_model_config(n_layers=2, d=128, n_heads_q=4, n_heads_kv=2, head_dim=64, ffn=256, vocab=512, eps=1e-6,
                               rope_theta=1e4, kv_block=32, kv_split=512, max_pos=256)
    w = _lib.bi_weights()
    h = ctypes.c_void_p()
    create = lambda: lib.bi_model_create(ctypes.byref(cfg), ctypes.byref(w), None, ctypes.byref(h))
    assert create() == bi.BI_ERR_UNSUPPORTED_SHAPE
    cfg.kv_block = 64
    cfg.kv_split = 100
    assert create() == bi.BI_ERR_INVALID_ARG
    cfg.kv_split = 512
    assert create() == bi.BI_ERR_INVALID_ARG   # null weight pointers
    assert "null" in bi.bi_last_error()


def test_workspace_queries_are_limit_sized(lib):
    cfg = _lib.bi_model_config(n_layers=4, d=512, n_heads_q=8, n_heads_kv=8, head_dim=64, ffn=1408, vocab=32000,
                               eps=1e-6, rope_theta=1e4, kv_block=64, kv_split=512, max_pos=1024)
    a = _lib.bi_forward_workspace_size(cfg, 1024, 16, 768, 512)
    b = _lib.bi_forward_workspace_size(cfg, 2048, 16, 768, 512)
    assert 0 < a < b
    assert _lib.bi_kv_cache_bytes(cfg, 10) == 4 * 10 * 8 * 64 * 64 * 2
    # invariant GEMM tile width depends on the weight shape only
    assert bi.bi_gemm_tile_n(32000, 512) == bi.bi_gemm_tile_n(32000, 512)
    assert bi.bi_gemm_workspace_size(16, 1536, 512, 0, bi.BI_INVARIANT) == 0
    assert bi.bi_gemm_workspace_size(16, 1536, 512, 0, bi.BI_FAST) > 0


@pytest.mark.skipif(__import__("torch").cuda.is_available(),
                    reason="passes dummy addresses; the refusal must be observed where nothing can launch")
def test_static_scratch_attention_refuses_oversized_calls_before_any_cuda_call(lib):
    # The size check of bi_attention_static_scratch runs on the host before any
    # CUDA call, so on a machine without a GPU a refused call returns
    # BI_ERR_INVALID_ARG, and a regressed check would show up as BI_ERR_CUDA
    # (no device), never as a launch.  Arguments: q T seq row0 pos0 P max_q_len
    # Hq Hkv hd k v block_table max_blk n_blocks max_ctx split scale out mode stream.
    def call(T, max_ctx, Hq=16, hd=128, mode=0):
        return lib.bi_attention_static_scratch(16, T, 16, 16, 16, 1, 64, Hq, 4, hd, 16, 16, 16, 1024, 1024, max_ctx,
                                               512, 0.088, 16, mode, None)
    # 64 rows x 16 heads x 128 splits x 130 x 4 bytes = 68 MB > 32 MiB
    assert call(64, 65536) == bi.BI_ERR_INVALID_ARG
    msg = bi.bi_last_error()
    assert "static scratch array holds 33554432 bytes" in msg and "68157440 bytes" in msg, msg
    # a product that does not fit in 64 bits is refused the same way (no wrap-around)
    assert call(1 << 40, 1 << 50) == bi.BI_ERR_INVALID_ARG
    assert "more than 2^64 bytes" in bi.bi_last_error()
    assert call(1 << 62, 1 << 62, Hq=1 << 30) == bi.BI_ERR_INVALID_ARG
    # bad mode and bad shapes are refused before the size check
    assert call(64, 4096, mode=3) == bi.BI_ERR_INVALID_ARG
    assert call(64, 4096, hd=0) == bi.BI_ERR_INVALID_ARG


def test_ssd_validation_without_gpu():
    lib = bi.load()
    assert bi.bi_ssd_state_bytes(4, 3, 64, 128, 64) == 0                      # H % G != 0
    assert bi.bi_ssd_state_bytes(4, 2, 64, 128, 64) == 4 * (4 * 128 * 64 + 64 * 4 * 128 + 64 * 4 * 64 + 64 * 4)
    args = [16, 16, 16, 16, 16, 16, 16, 1, 1]
    assert lib.bi_ssd_chunk_scan(*args, 4, 2, 64, 256, 64, 16, 1, 16, 0, None) == bi.BI_ERR_UNSUPPORTED_SHAPE
    assert lib.bi_ssd_chunk_scan(*args, 4, 3, 64, 128, 64, 16, 1, 16, 0, None) == bi.BI_ERR_INVALID_ARG
    assert lib.bi_ssd_chunk_scan(None, 16, 16, 16, 16, 16, 16, 0, 1, 4, 2, 64, 128, 64, 16, 1, 16, 0, None) == bi.BI_OK
    misaligned = [16, 16, 16, 16, 16, 16, 16, 1, 1, 4, 2, 64, 128, 64, 20, 1, 16, 0, None]   # state at byte 20
    assert lib.bi_ssd_chunk_scan(*misaligned) == bi.BI_ERR_INVALID_ARG


def test_product_path_does_not_reach_the_oracle():
    """The package (binding, decoder, build) imports neither the oracle nor the
    input generators: every step of the path runs in libbi.so (numpy serves the
    host bookkeeping only: index arrays, block tables)."""
    import ast
    pkg = os.path.join(ROOT, "invariant_forward_policy_gb300")
    for f in sorted(os.listdir(pkg)):
        if not f.endswith(".py"):
            continue
        tree = ast.parse(open(os.path.join(pkg, f)).read())
        for node in ast.walk(tree):
            names = []
            if isinstance(node, ast.Import):
                names = [a.name for a in node.names]
            elif isinstance(node, ast.ImportFrom) and node.level == 0:
                names = [node.module or ""]
            for n in names:
                assert n.split(".")[0] not in ("oracle", "synthetic"), (f, n)


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """Without libbi.so the first call raises; nothing falls back to the CPU."""
    monkeypatch.setattr(_lib, "_L", None)
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "libbi.so"))
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        _lib.load()
    with pytest.raises(RuntimeError):
        bi.bi_version()


def _header_no_comments():
    src = open(os.path.join(ROOT, "include", "bi.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return re.sub(r"//[^\n]*", "", src)


def _ctype_of(decl):
    """The ctypes type the binding must use for one C parameter / field / result type."""
    decl = " ".join(decl.replace("const", " ").split())
    if "*" in decl:
        return "char_p" if decl.startswith("char") and decl.count("*") == 1 else "ptr"
    base = decl.split()[0]
    return {"int64_t": ctypes.c_int64, "size_t": ctypes.c_size_t, "int": ctypes.c_int, "float": ctypes.c_float,
            "double": ctypes.c_double, "bi_status": ctypes.c_int, "void": None}[base]


def _same(want, got):
    if want == "ptr":
        return got is ctypes.c_void_p or (isinstance(got, type) and issubclass(got, ctypes._Pointer))
    if want == "char_p":
        return got is ctypes.c_char_p
    return got is want


def test_binding_types_match_the_header_prototypes():
    """Every ctypes signature has the header's arity and, parameter by parameter,
    the same width: a 32-bit int bound as 64 (or a pointer as an int) would be
    silent undefined behaviour."""
    src = _header_no_comments()
    protos = {}
    for m in re.finditer(r"([A-Za-z_][\w \*]*?)\b(bi_[a-z0-9_]+)\s*\(([^;{()]*)\)\s*;", src):
        res, name, args = m.group(1).strip(), m.group(2), m.group(3).strip()
        params = [] if args in ("", "void") else [a.strip() for a in args.split(",")]
        # drop the parameter name: the type is everything before the last identifier
        types = [re.sub(r"\b[A-Za-z_]\w*\s*$", "", p).strip() or p for p in params]
        protos[name] = (res, types)
    assert sorted(protos) == sorted(_lib._SIGS)
    for name, (res, types) in protos.items():
        want_res, want_args = _ctype_of(res), [_ctype_of(t) for t in types]
        got_res, got_args = _lib._SIGS[name]
        assert (want_res is None and got_res is None) or _same(want_res, got_res), (name, res, got_res)
        assert len(got_args) == len(want_args), (name, len(got_args), len(want_args))
        for i, (w, g) in enumerate(zip(want_args, got_args)):
            assert _same(w, g), (name, i, types[i], g)


def test_binding_structs_and_constants_match_the_header():
    src = _header_no_comments()
    for cls in (_lib.bi_model_config, _lib.bi_layer_weights, _lib.bi_weights):
        body = re.search(r"typedef struct \{([^}]*)\}\s*" + cls.__name__ + r"\s*;", src).group(1)
        fields = []
        for stmt in body.split(";"):
            stmt = stmt.strip()
            if not stmt:
                continue
            m = re.match(r"((?:const\s+)?[A-Za-z_]\w*\s*\**)\s*(.*)$", stmt)
            base, names = m.group(1), m.group(2)
            for nm in names.split(","):
                nm = nm.strip()
                stars = nm.count("*")
                fields.append((nm.strip("* "), _ctype_of(base + "*" * stars)))
        got = cls._fields_
        assert [f[0] for f in got] == [f[0] for f in fields], cls.__name__
        for (n, w), (_, g) in zip(fields, got):
            assert _same(w, g), (cls.__name__, n, g)
    for name, value in re.findall(r"\b(BI_[A-Z0-9_]+)\s*=\s*(\d+)", src):
        assert getattr(_lib, name) == int(value), name


_NULL_SWEEP = r"""
import ctypes, sys
sys.path.insert(0, sys.argv[1])
from invariant_forward_policy_gb300 import _lib
lib = _lib.load()
for name, (res, args) in _lib._SIGS.items():
    if name == "bi_device_status":          # synchronises the device
        continue
    for mode in (0, 1):
        vals = []
        for a in args:
            if a is _lib._vp or (isinstance(a, type) and issubclass(a, ctypes._Pointer)):
                vals.append(None)
            elif a in (_lib._f32, _lib._f64):
                vals.append(1.0)
            else:
                vals.append(mode)
        r = getattr(lib, name)(*vals)
        print(name, mode, r if isinstance(r, int) else "-")
"""


def test_every_entry_point_survives_null_pointers():
    """NULL pointers with zero sizes are no-ops; with non-zero sizes every call that
    returns a status refuses them (BI_ERR_INVALID_ARG or BI_ERR_UNSUPPORTED_SHAPE).
    Nothing crashes and nothing reaches the GPU."""
    import subprocess
    import sys
    r = subprocess.run([sys.executable, "-c", _NULL_SWEEP, ROOT], capture_output=True, text=True, timeout=300,
                       env=dict(os.environ, CUDA_VISIBLE_DEVICES=""))
    assert r.returncode == 0, r.stderr[-2000:]
    got = {}
    for line in r.stdout.split("\n"):
        if line.strip():
            name, mode, val = line.split()
            got[(name, int(mode))] = val
    not_status = {"bi_version", "bi_gemm_tile_n", "bi_device_status"}
    checked = 0
    for name, (res, args) in _lib._SIGS.items():
        if res is not ctypes.c_int or name in not_status:
            continue
        assert got[(name, 1)] in ("1", "2"), (name, got[(name, 1)])
        checked += 1
    assert checked >= 30
