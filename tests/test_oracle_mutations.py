"""The oracle's pins catch plausible mistakes.  Each case plants one slip (a
dropped term, a wrong sign or index, a transposed operand, a wrong block shape,
a tie broken the other way) in a temporary copy of `oracle/` and runs the pins
against that copy: they must fail.  An unmutated copy must pass (the harness
itself is sound).  Every mutation is made on the CPU, in the copy only."""
import concurrent.futures
import os
import shutil
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PINS = {
    "ops": ["test_oracle_pins.py"],
    "fp8": ["test_oracle_fp8_pins.py", "test_oracle_fp8_model_pins.py"],
    "ssd": ["test_oracle_ssd_pins.py"],
    "topk": ["test_oracle_topk_pins.py"],
}

# (module file, text to replace (exactly once), replacement, pin group)
MUTATIONS = [
    # RoPE: rotation direction, frequency exponent
    ("ops.py", "o1 = x1 * c - x2 * s", "o1 = x1 * c + x2 * s", "ops"),
    ("ops.py", "o2 = x2 * c + x1 * s", "o2 = x2 * c - x1 * s", "ops"),
    ("ops.py", "inv_freq = theta ** (-2.0 * i / head_dim)", "inv_freq = theta ** (-1.0 * i / head_dim)", "ops"),
    # RMSNorm: mean over d, the gain
    ("ops.py", "keepdims=True) / F32(d)", "keepdims=True) / F32(d + 1)", "ops"),
    ("ops.py", "y = round_bf16((r * inv) * np.asarray(gain, dtype=F32))", "y = round_bf16(r * inv)", "ops"),
    # linear layer off by a relative 1e-3
    ("ops.py", "c = np.matmul(a, b.T).astype(F32)", "c = (np.matmul(a, b.T) * 1.001).astype(F32)", "ops"),
    # attention: causal mask off by one, GQA head map, softmax scale
    ("ops.py", "mask = kpos[None, :] <= q_pos[r0:r1, None]", "mask = kpos[None, :] < q_pos[r0:r1, None] + 0.5 * (q_pos[r0:r1, None] == 0)", "ops"),
    ("ops.py", "kh = k[:, h // group, :]", "kh = k[:, h % k.shape[1], :]", "ops"),
    ("ops.py", "scale = F32(1.0) / np.sqrt(F32(hd), dtype=F32)", "scale = F32(1.0) / F32(hd)", "ops"),
    # SwiGLU sign, k3 sign
    ("ops.py", "silu = g / (F32(1.0) + np.exp(-g).astype(F32))", "silu = g / (F32(1.0) + np.exp(g).astype(F32))", "ops"),
    ("ops.py", "k3 = np.expm1(logr) - logr", "k3 = np.expm1(logr) + logr", "ops"),
    # decoder layer: residual into the FFN norm, gate and up swapped
    ("model.py", 'x, r = ops.rmsnorm(o, lw["ffn_norm"], shape.eps, residual=r)',
     'x, _ = ops.rmsnorm(o, lw["ffn_norm"], shape.eps)', "ops"),
    ("model.py", 'g = ops.linear(x, lw["w13"][:F])\n        u = ops.linear(x, lw["w13"][F:])',
     'u = ops.linear(x, lw["w13"][:F])\n        g = ops.linear(x, lw["w13"][F:])', "ops"),
    # MoE: combine weight of the wrong slot
    ("moe.py", "acc = acc + w[:, s: s + 1] * y[:, s, :]", "acc = acc + w[:, 0:1] * y[:, s, :]", "ops"),
    # bf16: round half up instead of half to even
    ("bf16.py", "r = (u + np.uint64(0x7FFF) + lsb) & np.uint64(0xFFFF0000)",
     "r = (u + np.uint64(0x8000)) & np.uint64(0xFFFF0000)", "ops"),
    # FP8: scale rounding, ties of the encoder, activation block shape, weight block shape
    ("fp8.py", "2.0 ** np.ceil(np.log2(amax[nz] / E4M3_MAX))", "2.0 ** np.floor(np.log2(amax[nz] / E4M3_MAX))", "fp8"),
    ("fp8.py", "(_POS_CODES[hi] % 2 == 0)", "(_POS_CODES[hi] % 2 == 1)", "fp8"),
    ("fp8.py", "return quantize_blocks(x, 1)", "return quantize_blocks(x, 128)", "fp8"),
    ("fp8.py", "return quantize_blocks(w, 128)", "return quantize_blocks(w, 1)", "fp8"),
    # FP8 decoder layer: K/V scales per token over all heads, V not round-tripped, K quantised before RoPE
    ("model.py", "q, s = ofp8.quantize_blocks(np.asarray(t, F32).reshape(n * h, hd), 1, block_cols=hd)\n"
                 "    return ofp8.dequantize_blocks(q, s, 1, block_cols=hd).reshape(n, h, hd)",
     "q, s = ofp8.quantize_blocks(np.asarray(t, F32).reshape(n, h * hd), 1, block_cols=h * hd)\n"
     "    return ofp8.dequantize_blocks(q, s, 1, block_cols=h * hd).reshape(n, h, hd)", "fp8"),
    ("model.py", "k, v = kv_round_trip(k), kv_round_trip(v)", "k = kv_round_trip(k)", "fp8"),
    ("model.py", "    k = ops.rope(k, pos, shape.rope_theta)\n    if w8:\n        k, v = kv_round_trip(k), kv_round_trip(v)",
     "    if w8:\n        k, v = kv_round_trip(k), kv_round_trip(v)\n    k = ops.rope(k, pos, shape.rope_theta)", "fp8"),
    # FP8 codes: subnormal exponent, the sign of zero
    ("fp8.py", "v[code] = sign * (m / 8.0) * 2.0 ** -6", "v[code] = sign * (m / 8.0) * 2.0 ** -7", "fp8"),
    ("fp8.py", "np.where(np.signbit(x), 0x80, 0)", "np.where(x < 0, 0x80, 0)", "fp8"),
    # logprob: target index, normaliser without the max, greedy ties to the highest id
    ("ops.py", "return x[np.arange(x.shape[0]), ids] - lse", "return x[np.arange(x.shape[0]), ids - 1] - lse", "ops"),
    ("ops.py", "lse = m[..., 0] + np.log(np.sum(np.exp(x - m), axis=-1))",
     "lse = np.log(np.sum(np.exp(x - m), axis=-1))", "ops"),
    ("ops.py", "return np.argmax(np.asarray(logits, dtype=F32), axis=-1).astype(np.int32)",
     "x = np.asarray(logits, dtype=F32)\n    return (x.shape[-1] - 1 - np.argmax(x[..., ::-1], axis=-1)).astype(np.int32)", "ops"),
    # acceptance statistics: sample std instead of the population std
    ("ops.py", '"std": float(d.std())', '"std": float(d.std(ddof=1)) if d.size > 1 else 0.0', "ops"),
    # MoE routing: ties to the highest expert id, normaliser of one slot only
    ("moe.py", 'order = np.argsort(-x, axis=1, kind="stable")[:, :k].astype(np.int32)',
     'order = (E - 1 - np.argsort(-x[:, ::-1], axis=1, kind="stable"))[:, :k].astype(np.int32)', "ops"),
    ("moe.py", "den = den + e[:, s: s + 1]", "den = den + e[:, 0:1]", "ops"),
    # scoring: rows shifted by one, no final norm
    ("model.py", "rows = np.arange(len(prompt) - 1, len(seq))", "rows = np.arange(len(prompt) - 2, len(seq) - 1)", "ops"),
    ("model.py", 'x, _ = ops.rmsnorm(r, w["final_norm"], shape.eps)\n    if return_layers:',
     'x = r\n    if return_layers:', "ops"),
    # Mamba-2: the entering state ignored
    ("ssd.py", "state = np.zeros((H, N, P)) if state0 is None else np.array(state0, np.float64)",
     "state = np.zeros((H, N, P))", "ssd"),
    # Mamba-2: decay applied after the input, group map, output read before the update
    ("ssd.py", "state[h] = np.exp(loga[t, h]) * state[h] + np.outer(B[t, g], x[t, h])",
     "state[h] = np.exp(loga[t, h]) * (state[h] + np.outer(B[t, g], x[t, h]))", "ssd"),
    ("ssd.py", "g = h // hpg", "g = h % n_groups", "ssd"),
    ("ssd.py", "state[h] = np.exp(loga[t, h]) * state[h] + np.outer(B[t, g], x[t, h])\n            y[t, h] = C[t, g] @ state[h]",
     "y[t, h] = C[t, g] @ state[h]\n            state[h] = np.exp(loga[t, h]) * state[h] + np.outer(B[t, g], x[t, h])", "ssd"),
    # Top-K: ties to the smaller position, output in ascending order, -0 below +0
    ("topk.py", "key=lambda p: (-float(s[p]), -p)", "key=lambda p: (-float(s[p]), p)", "topk"),
    ("topk.py", "chosen = sorted(cand[:k], reverse=True)", "chosen = sorted(cand[:k])", "topk"),
    ("topk.py", "key=lambda p: (-float(s[p]), -p)", "key=lambda p: (-float(s[p]), -np.copysign(1.0, s[p]), -p)", "topk"),
]


def _run_pins(oracle_dir, group):
    env = dict(os.environ)
    env["PYTHONPATH"] = os.pathsep.join([os.path.dirname(oracle_dir), ROOT])
    env["CUDA_VISIBLE_DEVICES"] = ""
    files = [os.path.join(ROOT, "tests", f) for f in PINS[group]]
    r = subprocess.run([sys.executable, "-m", "pytest", *files, "-x", "-q", "-m", "not gpu", "-p", "no:cacheprovider",
                        "--rootdir", ROOT], cwd=os.path.dirname(oracle_dir), env=env, capture_output=True, text=True,
                       timeout=600)
    return r.returncode, r.stdout[-1500:] + r.stderr[-500:]


def _copy(tmp, name):
    d = os.path.join(tmp, name, "oracle")
    shutil.copytree(os.path.join(ROOT, "oracle"), d, ignore=shutil.ignore_patterns("__pycache__"))
    return d


def _mutated_copy(tmp, i, mut):
    f, old, new, _ = mut
    d = _copy(tmp, f"m{i}")
    path = os.path.join(d, f)
    src = open(path).read()
    assert src.count(old) == 1, (f, old)
    open(path, "w").write(src.replace(old, new))
    return d


def test_unmutated_copy_passes_and_is_the_one_imported(tmp_path):
    d = _copy(str(tmp_path), "clean")
    for group in PINS:
        rc, out = _run_pins(d, group)
        assert rc == 0, (group, out)
    # the copy, not the tree's oracle, is what the pins import
    open(os.path.join(d, "topk.py"), "a").write("\nraise ImportError('copy imported')\n")
    rc, out = _run_pins(d, "topk")
    assert rc != 0 and "copy imported" in out


def test_pins_catch_every_planted_slip(tmp_path):
    tmp = str(tmp_path)
    dirs = [_mutated_copy(tmp, i, m) for i, m in enumerate(MUTATIONS)]
    workers = max(1, min(8, os.cpu_count() or 1))
    with concurrent.futures.ThreadPoolExecutor(workers) as ex:
        results = list(ex.map(lambda a: _run_pins(*a), [(d, m[3]) for d, m in zip(dirs, MUTATIONS)]))
    missed = [(m[0], m[2][:70]) for m, (rc, out) in zip(MUTATIONS, results) if rc != 1]
    assert not missed, missed
