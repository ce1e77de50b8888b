"""Pins of the oracle's fused producer step (RoPE + q concat + cache write)
against closed forms and against the already-pinned pieces of the oracle.

Source: "[ROCm][MLA][Perf] Fuse decode QK-RoPE + Q-concat + KV-concat +
KV-cache write for sparse MLA", Summary and Test plan: q_out =
concat(ql_nope, RoPE(q_pe)) in bf16 or as scaled_fp8_quant(., q_scale), and
the cache row concat_and_cache_mla(kv_c, RoPE(k_pe)). The rotation of a pair
(a, b) by theta is (a cos - b sin, b cos + a sin); neox pairs i with i + R/2,
GPT-J pairs 2i with 2i + 1.
"""
import numpy as np
import pytest
import torch

import oracle

DN, DR = 512, 64


def _bf16_bits(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _inputs(T, H, seed=0):
    g = np.random.default_rng(seed)
    ql = _bf16_bits(g.standard_normal((T, H, DN)))
    qp = _bf16_bits(g.standard_normal((T, H, DR)))
    kc = _bf16_bits(g.standard_normal((T, DN)))
    kp = _bf16_bits(g.standard_normal((T, DR)))
    return ql, qp, kc, kp


def _cos_sin(angles: np.ndarray) -> np.ndarray:
    """[P, DR] binary32 rows: cos of the DR/2 angles, then the sines."""
    return np.concatenate([np.cos(angles), np.sin(angles)], axis=1).astype(np.float32)


def _run(ql, qp, kc, kp, pos, cs, neox, slots, *, cache_fp8=False, q_fp8=False, q_scale=1.0, kv_scale=1.0,
         mode=1, num_slots=None):
    T = ql.shape[0]
    ns = num_slots if num_slots is not None else T
    cache = np.zeros((ns, DN + DR), dtype=np.uint8 if cache_fp8 else np.uint16)
    q_out, bad = oracle.fused_qk_rope_cache(ql, qp, kc, kp, pos, cs, neox, slots, cache, cache_fp8=cache_fp8,
                                            kv_scale=kv_scale, q_out_fp8=q_fp8, q_scale=q_scale, mode=mode)
    return q_out, cache, bad


@pytest.mark.parametrize("neox", [True, False])
def test_rope_f64_closed_forms(neox):
    g = np.random.default_rng(1)
    x = g.standard_normal(DR)
    # angle 0 is the identity
    assert np.array_equal(oracle.rope_f64(x, np.ones(DR // 2), np.zeros(DR // 2), neox), x)
    # a quarter turn maps each pair (a, b) to (-b, a)
    y = oracle.rope_f64(x, np.zeros(DR // 2), np.ones(DR // 2), neox)
    ia = np.arange(DR // 2) if neox else 2 * np.arange(DR // 2)
    ib = ia + DR // 2 if neox else ia + 1
    assert np.array_equal(y[ia], -x[ib]) and np.array_equal(y[ib], x[ia])
    # a rotation keeps each pair's length, and two rotations add their angles
    t1, t2 = g.uniform(-3, 3, DR // 2), g.uniform(-3, 3, DR // 2)
    r1 = oracle.rope_f64(x, np.cos(t1), np.sin(t1), neox)
    assert np.allclose(r1[ia] ** 2 + r1[ib] ** 2, x[ia] ** 2 + x[ib] ** 2, rtol=1e-13, atol=1e-13)
    r12 = oracle.rope_f64(r1, np.cos(t2), np.sin(t2), neox)
    assert np.allclose(r12, oracle.rope_f64(x, np.cos(t1 + t2), np.sin(t1 + t2), neox), rtol=1e-12, atol=1e-12)


def test_rope_gptj_is_neox_on_deinterleaved():
    """GPT-J on interleaved pairs equals neox on the de-interleaved vector."""
    g = np.random.default_rng(2)
    x = g.standard_normal(DR)
    t = g.uniform(-3, 3, DR // 2)
    perm = np.concatenate([np.arange(0, DR, 2), np.arange(1, DR, 2)])  # (2i, 2i+1) -> (i, i + R/2)
    neox = oracle.rope_f64(x[perm], np.cos(t), np.sin(t), True)
    gptj = oracle.rope_f64(x, np.cos(t), np.sin(t), False)
    back = np.empty(DR)
    back[perm] = neox
    assert np.array_equal(gptj, back)


@pytest.mark.parametrize("neox", [True, False])
@pytest.mark.parametrize("mode", [0, 1])
def test_producer_identity_and_quarter_turn(neox, mode):
    T, H = 3, 4
    ql, qp, kc, kp = _inputs(T, H)
    cs = _cos_sin(np.stack([np.zeros(DR // 2), np.full(DR // 2, np.pi / 2)]))
    cs[1, :DR // 2] = 0.0  # exact quarter turn (cos(pi/2) is not exactly 0 in binary32)
    cs[1, DR // 2:] = 1.0
    slots = np.array([2, 0, 1], dtype=np.int64)
    # position 0: the identity -> q_out == concat(ql_nope, q_pe), cache == concat(kv_c, k_pe)
    q_out, cache, bad = _run(ql, qp, kc, kp, np.zeros(T, np.int64), cs, neox, slots, mode=mode)
    assert bad == 0
    assert np.array_equal(q_out, np.concatenate([ql, qp], axis=2))
    assert np.array_equal(cache[slots], np.concatenate([kc, kp], axis=1))
    # position 1: the quarter turn, exact in bf16 -> the rope part is a signed permutation
    q_out, cache, bad = _run(ql, qp, kc, kp, np.ones(T, np.int64), cs, neox, slots, mode=mode)
    ia = np.arange(DR // 2) if neox else 2 * np.arange(DR // 2)
    ib = ia + DR // 2 if neox else ia + 1
    rope = q_out[:, :, DN:]
    assert np.array_equal(rope[:, :, ia], qp[:, :, ib] ^ np.uint16(0x8000))
    assert np.array_equal(rope[:, :, ib], qp[:, :, ia])
    assert np.array_equal(q_out[:, :, :DN], ql)
    krope = cache[slots][:, DN:]
    assert np.array_equal(krope[:, ia], kp[:, ib] ^ np.uint16(0x8000))
    assert np.array_equal(krope[:, ib], kp[:, ia])


@pytest.mark.parametrize("neox", [True, False])
def test_producer_bf16_is_the_rounded_rotation(neox):
    """Both modes give the fp64 rotation rounded to bf16: mode 0 exactly, mode 1
    (binary32 arithmetic) within one bf16 step, and equal almost everywhere."""
    T, H = 8, 16
    ql, qp, kc, kp = _inputs(T, H, seed=3)
    g = np.random.default_rng(4)
    cs = _cos_sin(g.uniform(-100, 100, (32, DR // 2)))
    pos = g.integers(0, 32, T)
    slots = np.arange(T, dtype=np.int64)
    q0, c0, _ = _run(ql, qp, kc, kp, pos, cs, neox, slots, mode=0)
    q1, c1, _ = _run(ql, qp, kc, kp, pos, cs, neox, slots, mode=1)
    # mode 0 against a direct fp64 rotation of each row, rounded to bf16 by torch (RNE)
    csd = cs.astype(np.float64)
    for t in range(T):
        c, s = csd[pos[t], :DR // 2], csd[pos[t], DR // 2:]
        for h in range(H):
            r = oracle.rope_f64(_bits_to_f64(qp[t, h]), c, s, neox)
            ref = torch.from_numpy(r).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
            assert np.array_equal(q0[t, h, DN:], ref), (t, h)
    diff = np.abs(_bits_to_f64(q1) - _bits_to_f64(q0))
    step = np.abs(_bits_to_f64(q0)) * 2.0 ** -7 + 1e-30
    assert np.all(diff <= step)
    assert np.mean(q1 == q0) > 0.99
    assert np.array_equal(c0[:, :DN], c1[:, :DN])


def test_producer_fp8_divides_by_the_scale():
    """fp8 q_out and cache rows are the codes of bf16 / scale (binary32
    division), the scaled_fp8_quant convention, with non-unit scales."""
    T, H = 4, 16
    ql, qp, kc, kp = _inputs(T, H, seed=5)
    g = np.random.default_rng(6)
    cs = _cos_sin(g.uniform(-10, 10, (8, DR // 2)))
    pos = g.integers(0, 8, T)
    slots = np.array([3, -1, 0, 1], dtype=np.int64)
    q_scale, kv_scale = np.float32(0.0137), np.float32(0.0211)
    qb, cb, bad = _run(ql, qp, kc, kp, pos, cs, True, slots, mode=1, num_slots=5)
    q8, c8, bad8 = _run(ql, qp, kc, kp, pos, cs, True, slots, mode=1, num_slots=5, q_fp8=True, cache_fp8=True,
                        q_scale=q_scale, kv_scale=kv_scale)
    assert bad == 0 and bad8 == 0
    xs = (qb.astype(np.uint32) << 16).view(np.float32)
    want = np.vectorize(lambda v: oracle.e4m3_encode(np.float32(v) / q_scale), otypes=[np.uint8])(xs)
    assert np.array_equal(q8, want)
    # with a non-unit scale, multiplying by it instead of dividing cannot alias
    mult = np.vectorize(lambda v: oracle.e4m3_encode(np.float32(v) * q_scale), otypes=[np.uint8])(xs)
    assert np.mean(mult == want) < 0.1
    # the cache rows equal the (pinned) cache-write oracle applied to the bf16 rows
    rows = slots >= 0
    ref = oracle.fp8_quantize(cb[slots[rows]], kv_scale)
    assert np.array_equal(c8[slots[rows]], ref)
    # slot -1 writes no row: slots 2 and 4 stay zero
    assert not c8[2].any() and not c8[4].any()


def test_producer_out_of_range_positions_and_slots():
    T, H = 4, 2
    ql, qp, kc, kp = _inputs(T, H, seed=7)
    cs = _cos_sin(np.zeros((4, DR // 2)))
    pos = np.array([0, 4, -1, 3], dtype=np.int64)   # 4 and -1 are outside [0, 4)
    slots = np.array([0, 1, 2, 9], dtype=np.int64)  # 9 is outside [0, 4)
    q_out, cache, bad = _run(ql, qp, kc, kp, pos, cs, True, slots, num_slots=4)
    assert bad == 3
    assert not q_out[1].any() and not q_out[2].any()   # tokens with a bad position: nothing written
    assert np.array_equal(q_out[3], np.concatenate([ql[3], qp[3]], axis=1))  # bad slot: q still written
    assert np.array_equal(cache[0], np.concatenate([kc[0], kp[0]]))
    assert not cache[1].any() and not cache[2].any() and not cache[3].any()
