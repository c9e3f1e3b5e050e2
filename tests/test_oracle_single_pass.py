"""The oracle's single-pass FC2 with online amax compensation ("miniTE
Technical Report" 5.6, Exploring Single-Pass Fusion), a research direction
the pages evaluate by its code differences from two-pass execution and its
compensation error.  Pins: with one K-tile it is the two-pass FC2; when a
row's max lies in its first tile every code is the two-pass code; the
compensated recurrence equals the direct sum of each tile's product at its
own outer scale; all-zero rows give zero.  The last test reports the
differences on rows shaped like the Qwen3 expert layer's FC2 input."""
import numpy as np

import oracle
import workloads


def _w2(rng, H=256, F=256):
    return oracle.quantize(workloads.gaussian_bf16(rng, (H, F), std=0.02), per_tensor=True)


def _two_pass(d, w2q):
    q = oracle.quantize(d)
    return q, oracle.gemm_f64(oracle.dequantize(*q), oracle.dequantize(*w2q, per_tensor=True))


def _close(y, ref, d, w2q):
    """Equal up to fp64 rounding order: within 1e-12 of sum_k |a_k b_k| (cancellation makes a
    relative test on the result itself meaningless near zero)."""
    q = oracle.quantize(d)
    bound = 1e-12 * oracle.abs_product_sum(oracle.dequantize(*q), oracle.dequantize(*w2q, per_tensor=True))
    return np.all(np.abs(y - ref) <= bound)


def test_one_tile_is_the_two_pass_fc2():
    rng = np.random.default_rng(1)
    d = workloads.gaussian_bf16(rng, (40, 256))
    w2q = _w2(rng)
    sp = oracle.fc2_single_pass(d, w2q, k_tile=256)
    q, y2 = _two_pass(d, w2q)
    assert np.array_equal(sp["codes"], q[0]) and np.array_equal(sp["sf"], q[1])
    assert np.array_equal(sp["gs_tiles"][:, 0].view(np.uint32), q[2].view(np.uint32))
    assert _close(sp["y_f64"], y2, d, w2q)


def test_max_in_the_first_tile_keeps_every_two_pass_code():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((32, 256)).astype(np.float32)
    x[:, 0] = 40.0 * np.sign(rng.standard_normal(32))  # the row max, in tile 0
    d = workloads.to_bf16_bits(x)
    w2q = _w2(rng)
    sp = oracle.fc2_single_pass(d, w2q, k_tile=64)
    q, y2 = _two_pass(d, w2q)
    assert np.array_equal(sp["codes"], q[0]) and np.array_equal(sp["sf"], q[1])
    assert np.all(sp["gs_tiles"] == q[2][:, None])
    assert _close(sp["y_f64"], y2, d, w2q)


def test_compensation_equals_each_tile_at_its_own_scale():
    """Rows whose magnitude grows tile by tile (the max in the last tile):
    every tile is encoded with a larger running amax than the one before, and
    O * gs_prev * gs_W2 must equal sum_i gs_i (A_i . B) gs_W2, A_i the tile's
    q s_b, computed directly from the returned codes and scales."""
    rng = np.random.default_rng(3)
    F, kt = 256, 64
    x = rng.standard_normal((24, F)).astype(np.float32) * np.repeat(2.0 ** np.arange(F // kt), kt)[None, :]
    d = workloads.to_bf16_bits(x)
    w2q = _w2(rng, F=F)
    sp = oracle.fc2_single_pass(d, w2q, k_tile=kt)
    gs = sp["gs_tiles"].astype(np.float64)
    assert np.all(np.diff(gs, axis=1) > 0)
    b = oracle.dequantize(w2q[0], w2q[1], np.ones(1, np.float32), per_tensor=True)
    direct = np.zeros_like(sp["y_f64"])
    for i in range(F // kt):
        c = slice(i * kt // 2, (i + 1) * kt // 2)
        s = slice(i * kt // 16, (i + 1) * kt // 16)
        a = oracle.dequantize(sp["codes"][:, c], sp["sf"][:, s], np.ones(len(d), np.float32))
        direct += gs[:, i:i + 1] * oracle.gemm_f64(a, b[:, i * kt:(i + 1) * kt])
    direct *= np.float64(w2q[2][0])
    assert _close(sp["y_f64"], direct, d, w2q)
    # the earlier tiles are coded against a smaller scale than the two-pass row scale
    q, _ = _two_pass(d, w2q)
    assert not np.array_equal(sp["codes"][:, :kt // 2], q[0][:, :kt // 2])
    assert np.array_equal(sp["gs_tiles"][:, -1].view(np.uint32), q[2].view(np.uint32))


def test_all_zero_rows_give_zero():
    rng = np.random.default_rng(4)
    d = workloads.gaussian_bf16(rng, (8, 256))
    d[3] = 0
    d[5, :128] = 0  # zero first tiles, then live
    sp = oracle.fc2_single_pass(d, _w2(rng), k_tile=64)
    assert not sp["y"][3].any() and not sp["codes"][3].any()
    assert sp["y"][5].any()


def test_single_pass_differences_on_expert_layer_rows():
    """FC2 inputs of a reduced Qwen3-shaped layer (H 2048, F 768, 8 experts,
    top-2), from the oracle's own chain: the single pass with 128-column
    K-tiles (FC1's N-tile of D) against two-pass execution and against the
    unquantized product of the same D."""
    rng = np.random.default_rng(5)
    T, E, k, H, F = 96, 8, 2, 2048, 768
    x = workloads.gaussian_bf16(rng, (T, H))
    logits = rng.standard_normal((T, E), dtype=np.float32)
    bias = rng.standard_normal(E, dtype=np.float32)
    w1 = [oracle.quantize(workloads.gaussian_bf16(rng, (2 * F, H), std=0.02), per_tensor=True) for _ in range(E)]
    w2 = [oracle.quantize(workloads.gaussian_bf16(rng, (H, F), std=0.02), per_tensor=True) for _ in range(E)]
    ref = oracle.moe_forward(x, logits, bias, w1, w2, k)
    off = ref["meta"]["off"]
    blocks_diff = n_blocks = 0
    e_sp = e_tp = e_between = norm = 0.0
    for e in range(E):
        lo, hi = int(off[e]), int(off[e + 1])
        if hi == lo:
            continue
        d = ref["D"][lo:hi]
        sp = oracle.fc2_single_pass(d, w2[e], k_tile=128)
        q, y2 = _two_pass(d, w2[e])
        cd = (sp["codes"].reshape(len(d), -1, 8) != q[0].reshape(len(d), -1, 8)).any(axis=2)
        blocks_diff += int((cd | (sp["sf"] != q[1])).sum())
        n_blocks += cd.size
        exact = oracle.gemm_f64(oracle.bf16_to_f64(d), oracle.dequantize(*w2[e], per_tensor=True))
        e_sp += float(np.sum((sp["y_f64"] - exact) ** 2))
        e_tp += float(np.sum((y2 - exact) ** 2))
        e_between += float(np.sum((sp["y_f64"] - y2) ** 2))
        norm += float(np.sum(exact ** 2))
    frac = blocks_diff / n_blocks
    rel_sp, rel_tp, rel_between = (np.sqrt(v / norm) for v in (e_sp, e_tp, e_between))
    print(f"\nsingle pass vs two pass: {frac:.2%} of {n_blocks} blocks coded differently; rel-L2 to the "
          f"unquantized product {rel_sp:.4e} (single) vs {rel_tp:.4e} (two-pass); between them {rel_between:.4e}")
    assert 0.0 < frac < 1.0
    assert rel_sp < 0.2 and rel_tp < 0.2 and rel_between < 0.2
