"""Mutation check of the oracle's pins (CPU only).

Each plausible mistake below (a dropped term, a wrong sign, index, axis,
rounding or order, a swapped operand) is planted in an in-memory copy of
the oracle's source; at least one pin of test_oracle_pins.py must then
fail.  The unmutated copy must pass them all, which checks the harness."""
import inspect
import itertools
import types

import pytest

import oracle.dsa_oracle as ORACLE
import test_oracle_pins as PINS

SRC = inspect.getsource(ORACLE)

# (what the mistake is, the oracle text it replaces, the mistaken text)
MUTANTS = [
    ("Hadamard without its 1/sqrt(n) scale",
     "@ (sylvester_hadamard(n) / np.sqrt(n))", "@ sylvester_hadamard(n)"),
    ("Sylvester recursion with the minus sign in the wrong block",
     "h = np.block([[h, h], [h, -h]])", "h = np.block([[h, -h], [h, h]])"),
    ("quantiser rounding half away from zero",
     "codes = np.where(sdiv > 0, np.rint(y), np.float32(0.0))",
     "codes = np.where(sdiv > 0, np.trunc(y + np.copysign(np.float32(0.5), y)), np.float32(0.0))"),
    ("quantiser dividing by the scale before its fp16 rounding",
     "sdiv = s16.astype(np.float32)[..., None]", "sdiv = s32[..., None]"),
    ("quantiser scale of absmax / 128",
     "s32 = amax / np.float32(127.0)", "s32 = amax / np.float32(128.0)"),
    ("int8 GEMM without the weight scale",
     "return acc * np.asarray(a_scale, dtype=F64)[:, None] * np.asarray(b_scale, dtype=F64)[None, :]",
     "return acc * np.asarray(a_scale, dtype=F64)[:, None]"),
    ("RoPE rotating the other way",
     "out[..., ia] = xa * c - xb * s", "out[..., ia] = xa * c + xb * s"),
    ("RoPE with the two pairings exchanged",
     "ia, ib = (2 * i, 2 * i + 1) if interleaved else (i, i + half)",
     "ia, ib = (i, i + half) if interleaved else (2 * i, 2 * i + 1)"),
    ("LayerNorm with the unbiased variance",
     "var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)",
     "var = ((x - mu) ** 2).sum(axis=-1, keepdims=True) / (x.shape[-1] - 1)"),
    ("LayerNorm with eps outside the square root",
     "return (x - mu) / np.sqrt(var + eps)", "return (x - mu) / (np.sqrt(var) + eps)"),
    ("indexer without the ReLU", "np.maximum(dots, 0.0)", "dots"),
    ("indexer without the key scale",
     "I = np.asarray(key_scale, F64) * (coef[:, None]", "I = (coef[:, None]"),
    ("indexer causal limit one key short",
     "I[np.arange(keys.shape[0]) > pos_t] = -np.inf", "I[np.arange(keys.shape[0]) >= pos_t] = -np.inf"),
    ("top-k taking the smallest scores",
     "order = np.lexsort((np.arange(n_valid), -s))", "order = np.lexsort((np.arange(n_valid), s))"),
    ("top-k breaking ties towards the larger index",
     "order = np.lexsort((np.arange(n_valid), -s))", "order = np.lexsort((-np.arange(n_valid), -s))"),
    ("attention without the softmax scale", "S = scale * (q @ kv.T)", "S = q @ kv.T"),
    ("attention values from the last d_v dims",
     "out = (p @ kv[:, :d_v]) / l", "out = (p @ kv[:, -d_v:]) / l"),
    ("attention sink left out of the denominator",
     "l = l + np.exp(sk[:, None] - m)", "l = l"),
    ("attention sink term not shifted by the running max",
     "l = l + np.exp(sk[:, None] - m)", "l = l + np.exp(sk[:, None])"),
    ("attention lse without the max added back",
     "return out, (m + np.log(l))[:, 0]", "return out, np.log(l)[:, 0]"),
    ("attention max ignoring the sink",
     "m = np.maximum(m, sk[:, None])", "m = m"),
    ("power-of-two scale rounded down",
     "up = np.where(m == 0.5, e - 1, e).astype(np.int32)", "up = (e - 1).astype(np.int32)"),
    ("mHC rounds normalising columns before rows",
     "        c = c / (c.sum(axis=-1, keepdims=True) + eps)\n        c = c / (c.sum(axis=-2, keepdims=True) + eps)",
     "        c = c / (c.sum(axis=-2, keepdims=True) + eps)\n        c = c / (c.sum(axis=-1, keepdims=True) + eps)"),
    ("mHC pre and post scales exchanged",
     "np.full(hc, hc_scale[0]), np.full(hc, hc_scale[1])", "np.full(hc, hc_scale[1]), np.full(hc, hc_scale[0])"),
    ("mHC post gate without its factor 2",
     "post = 2.0 * sig(z[:, hc:2 * hc])", "post = sig(z[:, hc:2 * hc])"),
    ("mHC softmax without eps", "c = c / c.sum(axis=-1, keepdims=True) + eps", "c = c / c.sum(axis=-1, keepdims=True)"),
    ("RMSNorm over the sum of squares instead of the mean",
     "x / np.sqrt((x * x).mean(axis=-1, keepdims=True) + eps)",
     "x / np.sqrt((x * x).sum(axis=-1, keepdims=True) + eps)"),
    ("MLA query with its two parts in the other order",
     "return np.concatenate([q_abs, q_pe], axis=-1)", "return np.concatenate([q_pe, q_abs], axis=-1)"),
    ("MLA head rows read with the rotary dims first",
     "u[..., :MLA_D_N], np.asarray(w_uk, dtype=F64))", "u[..., MLA_D_R:], np.asarray(w_uk, dtype=F64))"),
    ("MLA latent row without its RMSNorm",
     "lat = rms_norm(c[:, :MLA_D_C], gamma_kv, eps)", "lat = c[:, :MLA_D_C] * np.asarray(gamma_kv, F64)"),
    ("MLA latent row with its two parts in the other order",
     "return np.concatenate([lat, pe], axis=-1)", "return np.concatenate([pe, lat], axis=-1)"),
    ("paged rows offset by the block number instead of the row in the block",
     "return blk * inp.block_size + s % inp.block_size", "return blk * inp.block_size + s // inp.block_size"),
    ("k stream without its Hadamard transform",
     "k, k_scale = dynamic_quant(hadamard_rows(kr))", "k, k_scale = dynamic_quant(kr)"),
    ("LayerNorm without beta",
     "/ np.sqrt(var + eps) * np.asarray(gamma, F64) + np.asarray(beta, F64)",
     "/ np.sqrt(var + eps) * np.asarray(gamma, F64)"),
    ("weight stream without w_scale", "* float(p.w_scale)).astype(np.float32)", ").astype(np.float32)"),
    ("q stream without RoPE",
     "qr = rope(qf, p.pos, p.rope_cos, p.rope_sin, p.d_rope, bool(p.rope_interleaved))", "qr = qf"),
    ("key-cache scale taken from the first token",
     "k_scale_cache[p.slot[t]] = k_scale[t]", "k_scale_cache[p.slot[t]] = k_scale[0]"),
    ("act_quant dividing in float64 instead of the page's fp32",
     "        y = x32 / sd\n", "        y = x32.astype(np.float64) / sd\n"),
    ("int8 GEMM output left in fp32",
     "return int8_gemm_dequant(a, a_scale, b, b_scale).astype(np.float16)",
     "return int8_gemm_dequant(a, a_scale, b, b_scale).astype(np.float32)"),
    ("attention lse without the running maximum",
     "return out, (m + np.log(l))[:, 0]", "return out, (np.log(l))[:, 0]"),
    ("top-k padded with 0 instead of -1",
     "out = np.full(k, -1, dtype=np.int64)", "out = np.zeros(k, dtype=np.int64)"),
    ("indexer weights without the q scale",
     "coef = np.asarray(w_tok, F64) * np.asarray(q_scale_tok, F64)", "coef = np.asarray(w_tok, F64)"),
    ("attention sink ignored when nothing is selected",
     "return np.zeros((H, d_v)), (np.full(H, -np.inf) if sk is None else sk.copy())",
     "return np.zeros((H, d_v)), np.full(H, -np.inf)"),
    ("mHC pre gate without eps", "pre = sig(z[:, :hc]) + eps", "pre = sig(z[:, :hc])"),
    ("mHC first column step without eps",
     "c = c / c.sum(axis=-1, keepdims=True) + eps\n    c = c / (c.sum(axis=-2, keepdims=True) + eps)",
     "c = c / c.sum(axis=-1, keepdims=True) + eps\n    c = c / c.sum(axis=-2, keepdims=True)"),
    ("RMSNorm without eps",
     "x / np.sqrt((x * x).mean(axis=-1, keepdims=True) + eps)", "x / np.sqrt((x * x).mean(axis=-1, keepdims=True))"),
    ("MLA query latent without gamma_q",
     "c_q = rms_norm(x @ bf16_bits_to_f64(p.w_dq).T, p.gamma_q, p.rms_eps)",
     "c_q = rms_norm(x @ bf16_bits_to_f64(p.w_dq).T, np.ones_like(p.gamma_q), p.rms_eps)"),
    ("MLA latent row without gamma_kv",
     "lat = rms_norm(c[:, :MLA_D_C], gamma_kv, eps)", "lat = rms_norm(c[:, :MLA_D_C], np.ones_like(gamma_kv), eps)"),
    ("MLA query rotated one position late",
     "q_pe = rope(u[..., MLA_D_N:], pos, cos_tab, sin_tab, MLA_D_R, interleaved)",
     "q_pe = rope(u[..., MLA_D_N:], np.asarray(pos) + 1, cos_tab, sin_tab, MLA_D_R, interleaved)"),
    ("MLA up-projection without the q_lora scale",
     "u = int8_gemm_dequant(q_lora, q_lora_scale, w_uq, w_uq_scale)",
     "u = int8_gemm_dequant(q_lora, np.ones_like(q_lora_scale), w_uq, w_uq_scale)"),
    ("attention taking index -1 as row 0", "idx = idx[idx >= 0]", "idx = np.where(idx >= 0, idx, 0)"),
    ("mHC one Sinkhorn round too many", "for _ in range(iters):", "for _ in range(iters + 1):"),
    ("RMSNorm with eps outside the root",
     "x / np.sqrt((x * x).mean(axis=-1, keepdims=True) + eps)",
     "x / (np.sqrt((x * x).mean(axis=-1, keepdims=True)) + eps)"),
    ("LayerNorm without centring the numerator",
     "return (x - mu) / np.sqrt(var + eps)", "return x / np.sqrt(var + eps)"),
    ("act_quant scale stored through fp16",
     "return codes.astype(np.int8), s.astype(np.float32)",
     "return codes.astype(np.int8), s.astype(np.float16).astype(np.float32)"),
    ("power-of-two scale one step up when it already is one",
     "up = np.where(m == 0.5, e - 1, e).astype(np.int32)", "up = e.astype(np.int32)"),
    ("int8 GEMM with one activation scale for every row",
     "return acc * np.asarray(a_scale, dtype=F64)[:, None] * np.asarray(b_scale, dtype=F64)[None, :]",
     "return acc * np.asarray(a_scale, dtype=F64).mean() * np.asarray(b_scale, dtype=F64)[None, :]"),
    ("attention sink in log2 units", "l = l + np.exp(sk[:, None] - m)", "l = l + np.exp2(sk[:, None] - m)"),
    ("mHC comb logits scaled by the post scale", "np.full(hc * hc, hc_scale[2])", "np.full(hc * hc, hc_scale[1])"),
    ("MLA query rotary dims not rotated",
     "q_pe = rope(u[..., MLA_D_N:], pos, cos_tab, sin_tab, MLA_D_R, interleaved)", "q_pe = u[..., MLA_D_N:]"),
    ("MLA latent row rotary dims not rotated",
     "pe = rope(c[:, None, MLA_D_C:], pos, cos_tab, sin_tab, MLA_D_R, interleaved)[:, 0, :]", "pe = c[:, MLA_D_C:]"),
    ("Hadamard applied twice",
     "return np.asarray(x, dtype=F64) @ (sylvester_hadamard(n) / np.sqrt(n))",
     "return np.asarray(x, dtype=F64) @ (sylvester_hadamard(n) / np.sqrt(n)) @ (sylvester_hadamard(n) / np.sqrt(n))"),
]


def _module(src: str) -> types.ModuleType:
    m = types.ModuleType("oracle_mutant")
    exec(compile(src, "oracle_mutant", "exec"), m.__dict__)
    return m


def _pin_calls():
    """Every pin as (name, zero-argument callable), parametrised pins once per
    combination of their parameters."""
    calls = []
    for name, fn in sorted(vars(PINS).items()):
        if not (name.startswith("test_") and callable(fn)):
            continue
        marks = [m for m in getattr(fn, "pytestmark", []) if m.name == "parametrize"]
        if not marks:
            calls.append((name, fn))
            continue
        names, grids = [], []
        for m in marks:
            argnames = m.args[0]
            argnames = [a.strip() for a in argnames.split(",")] if isinstance(argnames, str) else list(argnames)
            values = [v if len(argnames) > 1 else (v,) for v in m.args[1]]
            names.append(argnames)
            grids.append(values)
        for combo in itertools.product(*grids):
            kw = {}
            for argnames, vals in zip(names, combo):
                kw.update(dict(zip(argnames, vals)))
            calls.append((f"{name}{kw}", lambda fn=fn, kw=kw: fn(**kw)))
    return calls


def _failing_pin(module, monkeypatch):
    monkeypatch.setattr(PINS, "O", module)
    for name, call in _pin_calls():
        try:
            call()
        except Exception:  # an assertion, or a shape error the mistake causes
            return name
    return None


def test_unmutated_copy_passes_every_pin(monkeypatch):
    assert _failing_pin(_module(SRC), monkeypatch) is None


@pytest.mark.filterwarnings("ignore::RuntimeWarning")  # a mistaken oracle may overflow
@pytest.mark.parametrize("what,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_fails_a_pin(what, old, new, monkeypatch):
    assert SRC.count(old) == 1, f"the oracle text for '{what}' is not unique"
    caught = _failing_pin(_module(SRC.replace(old, new)), monkeypatch)
    assert caught is not None, f"no pin fails when the oracle has: {what}"
