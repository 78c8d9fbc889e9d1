"""Pins for the CPU oracle (no GPU).

The oracle (oracle/attn_oracle.c, oracle/online.py) is checked against things
other than itself:
  * the library routine torch.nn.functional.scaled_dot_product_attention and
    torch.logsumexp, both in float64 on the CPU;
  * brute force with exactly rounded sums (math.fsum) on tiny inputs;
  * closed forms: constant V rows, one dominant key, zero scale, rows of P
    summing to one, joint permutation of the key/value rows, duplication of
    all key/value rows (LSE + ln 2), a per-row constant added to the scores;
  * the worked numbers printed in "B200 Attention Kernel from Scratch to
    Near-SOTA in 60 Diagrams" (tests/golden/worked_values.txt).
Each plausible slip in the oracle (a dropped scale, a wrong sign, a missing
normalisation, a wrong head offset when Sq != Sk, an LSE without the max)
fails at least one of these.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import online
from dense_attention_forward_attn_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append([c.strip() for c in line.split("|")])
    return rows


def _f64(bits):
    return torch.from_numpy(online.bf16_bits_to_f64(bits))


def _sdpa(qb, kb, vb, scale):
    q, k, v = _f64(qb), _f64(kb), _f64(vb)
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, scale=scale)
    lse = torch.logsumexp(scale * (q @ k.transpose(-1, -2)), dim=-1)
    return o.numpy(), lse.numpy()


SHAPES = [  # B, H, Sq, Sk, D
    (1, 2, 64, 80, 128),
    (2, 3, 33, 17, 16),
    (1, 1, 128, 128, 128),
    (2, 2, 5, 300, 8),
]


def test_worked_values_table():
    for name, expr, printed, tol, _where in _read_table("worked_values.txt"):
        got = eval(expr, {"math": math})
        assert abs(got - float(printed)) <= float(tol), (name, got, printed)


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("seed", [0, 7])
def test_oracle_matches_library_sdpa_f64(shape, seed):
    B, H, Sq, Sk, D = shape
    qb, kb, vb = wl.make_inputs_bits(B, H, Sq, Sk, D, seed=seed)
    scale = 1.0 / math.sqrt(D)
    o, lse = oracle.attn_fwd(qb, kb, vb, scale)
    o_ref, lse_ref = _sdpa(qb, kb, vb, scale)
    np.testing.assert_allclose(o, o_ref, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-12, atol=1e-12)


def test_oracle_matches_library_on_stress_distribution():
    qb, kb, vb = wl.make_inputs_bits(1, 2, 96, 256, 128, seed=3, qk_std=3.0,
                                     spike_every=64, spike_factor=8.0)
    scale = 1.0 / math.sqrt(128)
    o, lse = oracle.attn_fwd(qb, kb, vb, scale)
    o_ref, lse_ref = _sdpa(qb, kb, vb, scale)
    np.testing.assert_allclose(o, o_ref, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-12, atol=1e-10)


def test_oracle_matches_fsum_bruteforce():
    B, H, Sq, Sk, D = 1, 2, 5, 7, 16
    qb, kb, vb = wl.make_inputs_bits(B, H, Sq, Sk, D, seed=11, qk_std=2.0)
    scale = 0.3
    q, k, v = (online.bf16_bits_to_f64(x) for x in (qb, kb, vb))
    o, lse = oracle.attn_fwd(qb, kb, vb, scale)
    for h in range(H):
        for i in range(Sq):
            s = [scale * math.fsum(q[0, h, i, d] * k[0, h, j, d] for d in range(D)) for j in range(Sk)]
            m = max(s)
            e = [math.exp(x - m) for x in s]
            l = math.fsum(e)
            for d in range(D):
                ref = math.fsum(e[j] * v[0, h, j, d] for j in range(Sk)) / l
                assert abs(o[0, h, i, d] - ref) <= 1e-14 * max(1.0, abs(ref))
            assert abs(lse[0, h, i] - (m + math.log(l))) <= 1e-14 * max(1.0, abs(m))


def test_constant_value_rows_give_that_row():
    qb, kb, _ = wl.make_inputs_bits(1, 2, 40, 50, 32, seed=1)
    c = np.linspace(-2, 2, 32, dtype=np.float32)
    vb = np.broadcast_to(wl.to_bf16_bits(c), (1, 2, 50, 32)).copy()
    o, _ = oracle.attn_fwd(qb, kb, vb, 0.25)
    np.testing.assert_allclose(o, np.broadcast_to(wl.bf16_bits_to_f32(vb[0, 0, 0]), o.shape),
                               rtol=0, atol=1e-14)


def test_single_dominant_key_copies_its_value_row():
    D, Sk = 16, 64
    qb, kb, vb = wl.make_inputs_bits(1, 1, 8, Sk, D, seed=2)
    q = np.ones((1, 1, 8, D), np.float32)
    k = wl.bf16_bits_to_f32(kb).copy()
    k = np.clip(k, -1, 1)
    jstar = 37
    k[0, 0, jstar, :] = 8.0          # score of j* = 128*scale, others <= 16*scale
    scale = 1.0
    qb, kb = wl.to_bf16_bits(q), wl.to_bf16_bits(k)
    o, lse = oracle.attn_fwd(qb, kb, vb, scale)
    v = wl.bf16_bits_to_f32(vb)
    np.testing.assert_allclose(o[0, 0], np.broadcast_to(v[0, 0, jstar], (8, D)), atol=0,
                               rtol=1e-12)
    np.testing.assert_allclose(lse, 128.0, rtol=1e-14)


def test_zero_scale_is_uniform_average():
    qb, kb, vb = wl.make_inputs_bits(2, 2, 16, 48, 32, seed=5)
    o, lse = oracle.attn_fwd(qb, kb, vb, 0.0)
    v = online.bf16_bits_to_f64(vb)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(axis=2, keepdims=True), o.shape),
                               rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse, math.log(48), rtol=1e-14)


def test_probability_rows_sum_to_one_and_weight_values():
    qb, kb, vb = wl.make_inputs_bits(1, 1, 20, 30, 64, seed=9, qk_std=2.0)
    scale = 0.125
    p = oracle.attn_probs(qb[0, 0], kb[0, 0], scale)
    assert (p >= 0).all()
    np.testing.assert_allclose(p.sum(axis=1), 1.0, rtol=0, atol=1e-14)
    o, _ = oracle.attn_fwd(qb, kb, vb, scale)
    np.testing.assert_allclose(o[0, 0], p @ online.bf16_bits_to_f64(vb[0, 0]), rtol=1e-12, atol=1e-14)


def test_joint_permutation_of_keys_and_values():
    qb, kb, vb = wl.make_inputs_bits(1, 2, 24, 64, 32, seed=4)
    perm = np.random.Generator(np.random.PCG64(0)).permutation(64)
    o1, l1 = oracle.attn_fwd(qb, kb, vb, 0.2)
    o2, l2 = oracle.attn_fwd(qb, kb[:, :, perm], vb[:, :, perm], 0.2)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(l1, l2, rtol=1e-14)


def test_duplicated_keys_and_values_add_ln2():
    qb, kb, vb = wl.make_inputs_bits(1, 2, 24, 40, 32, seed=6)
    o1, l1 = oracle.attn_fwd(qb, kb, vb, 0.2)
    o2, l2 = oracle.attn_fwd(qb, np.concatenate([kb, kb], axis=2), np.concatenate([vb, vb], axis=2), 0.2)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(l2 - l1, math.log(2.0), rtol=0, atol=1e-12)


def test_per_row_constant_added_to_scores_only_shifts_lse():
    # k_j -> k_j + u for every key j adds scale*q_i.u to every score of row i.
    # Small integers keep every value exact in BF16.
    rng = np.random.Generator(np.random.PCG64(1))
    q = rng.integers(-3, 4, size=(1, 1, 12, 8)).astype(np.float32)
    k = rng.integers(-3, 4, size=(1, 1, 20, 8)).astype(np.float32)
    v = rng.standard_normal((1, 1, 20, 8), dtype=np.float32)
    u = rng.integers(-2, 3, size=8).astype(np.float32)
    scale = 0.5
    qb, kb, kub, vb = (wl.to_bf16_bits(x) for x in (q, k, k + u, v))
    o1, l1 = oracle.attn_fwd(qb, kb, vb, scale)
    o2, l2 = oracle.attn_fwd(qb, kub, vb, scale)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(l2 - l1, scale * (q[0, 0] @ u)[None, None], rtol=0, atol=1e-12)


def test_selected_rows_equal_full_forward():
    qb, kb, vb = wl.make_inputs_bits(2, 3, 40, 56, 32, seed=8)
    o, lse = oracle.attn_fwd(qb, kb, vb, 0.17)
    rng = np.random.Generator(np.random.PCG64(2))
    bh = rng.integers(0, 6, 25)
    rows = rng.integers(0, 40, 25)
    o_r, l_r = oracle.attn_fwd_rows(qb, kb, vb, 0.17, bh, rows)
    np.testing.assert_array_equal(o_r, o.reshape(6, 40, 32)[bh, rows])
    np.testing.assert_array_equal(l_r, lse.reshape(6, 40)[bh, rows])


def test_rows_rejects_out_of_range_index():
    qb, kb, vb = wl.make_inputs_bits(1, 1, 4, 4, 8, seed=0)
    with pytest.raises(RuntimeError):
        oracle.attn_fwd_rows(qb, kb, vb, 1.0, [0], [4])


# ---------------------------------------------------------------- online recurrence

@pytest.mark.parametrize("block_n", [1, 7, 64, 128])
def test_online_recurrence_reaches_plain_definition(block_n):
    qb, kb, vb = wl.make_inputs_bits(1, 2, 32, 384, 128, seed=12, qk_std=3.0,
                                     spike_every=64, spike_factor=8.0)
    scale = 1.0 / math.sqrt(128)
    o, lse = oracle.attn_fwd(qb, kb, vb, scale)
    o2, lse2, reb = online.online_attention(qb, kb, vb, scale, block_n=block_n)
    np.testing.assert_allclose(o2, o, rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(lse2, lse, rtol=1e-12, atol=1e-10)
    assert (reb >= 1).all()


@pytest.mark.parametrize("split", [128, 384, 640])
def test_kv_split_combine_reproduces_the_whole_softmax(split):
    """The reading the split schedule follows: an item's KV range cut into [0, x) and [x, n), each
    part run through the pages' online recurrence on its own (its own kept max and row sum), then
    combined with L_i = m_i + log2 l_i, L = log2(2^L0 + 2^L1), O = sum_i 2^(L_i - L) O_i / l_i,
    equals the softmax over all keys, and L ln 2 is its LSE."""
    qb, kb, vb = wl.make_inputs_bits(1, 1, 96, 768, 128, seed=12, qk_std=2.0)
    scale = 1.0 / math.sqrt(128)
    q, k, v = (online.bf16_bits_to_f64(x)[0, 0] for x in (qb, kb, vb))
    parts = []
    for lo, hi in ((0, split), (split, 768)):
        o_i, _, _, m_i, l_i = online.online_attention_head(q, k[lo:hi], v[lo:hi], scale)
        parts.append((o_i, m_i + np.log2(l_i)))
    L = np.logaddexp2(parts[0][1], parts[1][1])
    o = sum(np.exp2(L_i - L)[:, None] * o_i for o_i, L_i in parts)
    o_ref, lse_ref = oracle.attn_fwd(qb, kb, vb, scale)
    assert np.abs(o - o_ref[0, 0]).max() <= 1e-12
    assert np.abs(L * math.log(2.0) - lse_ref[0, 0]).max() <= 1e-12


def test_online_recurrence_threshold_never_and_always():
    qb, kb, vb = wl.make_inputs_bits(1, 1, 16, 512, 64, seed=13, qk_std=2.0)
    scale = 0.125
    o, lse = oracle.attn_fwd(qb, kb, vb, scale)
    for thr in (0.0, 1e300):   # rebase on every increase / only on the first tile
        o2, lse2, reb = online.online_attention(qb, kb, vb, scale, block_n=32, threshold_log2=thr)
        np.testing.assert_allclose(o2, o, rtol=1e-9, atol=1e-12)
        np.testing.assert_allclose(lse2, lse, rtol=1e-12, atol=1e-10)
    assert (reb == 1).all()


def _two_tile_row(gap_log2, threshold=online.REBASE_THRESHOLD_LOG2):
    # scale = ln 2 makes scale*log2(e) = 1, so raw scores are already base-2 units.
    q = np.array([[1.0]])
    k = np.array([[0.0], [gap_log2]])
    v = np.array([[1.0], [2.0]])
    return online.online_attention_head(q, k, v, math.log(2.0), block_n=1, threshold_log2=threshold)


def _golden(name):
    for row in _read_table("worked_values.txt"):
        if row[0] == name:
            return float(row[2]), float(row[3])
    raise KeyError(name)


def test_online_gap_below_threshold_keeps_stale_max():
    printed, tol = _golden("exp2_gap_7_78")
    o, lse, reb, m_kept, rowsum = _two_tile_row(7.78)
    assert reb[0] == 1 and m_kept[0] == 0.0            # no rebase on the second tile
    assert abs((rowsum[0] - 1.0) - printed) <= tol      # the new max entered as P ~= 219
    np.testing.assert_allclose(lse, np.log(1.0 + 2.0 ** 7.78), rtol=1e-14)
    np.testing.assert_allclose(o[0, 0], (1.0 + 2.0 * 2.0 ** 7.78) / (1.0 + 2.0 ** 7.78), rtol=1e-14)


def test_online_gap_at_threshold_rebases():
    printed, _ = _golden("exp2_threshold")
    o, lse, reb, m_kept, rowsum = _two_tile_row(8.0)
    assert reb[0] == 2 and m_kept[0] == 8.0             # ">=" rebases
    assert rowsum[0] == 1.0 + 1.0 / printed             # old row sum rescaled by 1/256


def test_online_gap_20_without_rebase_grows_p():
    printed, _ = _golden("exp2_gap_20")
    o, lse, reb, m_kept, rowsum = _two_tile_row(20.0, threshold=1e300)
    assert reb[0] == 1 and rowsum[0] - 1.0 == printed   # largest P = 1,048,576
    np.testing.assert_allclose(lse, np.log(1.0 + 2.0 ** 20), rtol=1e-14)


# ---------------------------------------------------------------- causal (top-left aligned)

def _sdpa_causal(qb, kb, vb, scale):
    q, k, v = _f64(qb), _f64(kb), _f64(vb)
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, scale=scale, is_causal=True)
    Sq, Sk = q.shape[2], k.shape[2]
    mask = torch.ones(Sq, Sk, dtype=torch.bool).tril(diagonal=0)
    s = (scale * (q @ k.transpose(-1, -2))).masked_fill(~mask, float("-inf"))
    return o.numpy(), torch.logsumexp(s, dim=-1).numpy()


@pytest.mark.parametrize("shape", [(1, 2, 64, 64, 128), (2, 1, 40, 90, 16), (1, 2, 90, 40, 16),
                                   (1, 1, 130, 130, 32)])
def test_causal_oracle_matches_library_sdpa_f64(shape):
    B, H, Sq, Sk, D = shape
    qb, kb, vb = wl.make_inputs_bits(B, H, Sq, Sk, D, seed=31)
    scale = 1.0 / math.sqrt(D)
    o, lse = oracle.attn_fwd(qb, kb, vb, scale, causal=True)
    o_ref, lse_ref = _sdpa_causal(qb, kb, vb, scale)
    np.testing.assert_allclose(o, o_ref, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-12, atol=1e-12)


def test_causal_oracle_matches_fsum_bruteforce():
    B, H, Sq, Sk, D = 1, 1, 6, 4, 8
    qb, kb, vb = wl.make_inputs_bits(B, H, Sq, Sk, D, seed=32, qk_std=2.0)
    q, k, v = (online.bf16_bits_to_f64(x)[0, 0] for x in (qb, kb, vb))
    o, lse = oracle.attn_fwd(qb, kb, vb, 0.5, causal=True)
    for i in range(Sq):
        keys = range(min(i + 1, Sk))
        s = [0.5 * math.fsum(q[i, d] * k[j, d] for d in range(D)) for j in keys]
        m = max(s)
        e = [math.exp(x - m) for x in s]
        l = math.fsum(e)
        for d in range(D):
            ref = math.fsum(e[n] * v[j, d] for n, j in enumerate(keys)) / l
            assert abs(o[0, 0, i, d] - ref) <= 1e-14 * max(1.0, abs(ref))
        assert abs(lse[0, 0, i] - (m + math.log(l))) <= 1e-14 * max(1.0, abs(m))


def test_causal_closed_forms():
    qb, kb, vb = wl.make_inputs_bits(1, 2, 50, 30, 16, seed=33)
    o_c, l_c = oracle.attn_fwd(qb, kb, vb, 0.4, causal=True)
    o_n, l_n = oracle.attn_fwd(qb, kb, vb, 0.4)
    v = online.bf16_bits_to_f64(vb)
    q, k = online.bf16_bits_to_f64(qb), online.bf16_bits_to_f64(kb)
    # row 0 sees only key 0
    np.testing.assert_allclose(o_c[:, :, 0], v[:, :, 0], rtol=0, atol=1e-15)
    np.testing.assert_allclose(l_c[:, :, 0], 0.4 * (q[:, :, 0] * k[:, :, 0]).sum(-1), rtol=1e-14)
    # rows at or past the last key see every key
    np.testing.assert_array_equal(o_c[:, :, 29:], o_n[:, :, 29:])
    np.testing.assert_array_equal(l_c[:, :, 29:], l_n[:, :, 29:])
    p = oracle.attn_probs(qb[0, 0], kb[0, 0], 0.4, causal=True)
    assert (np.triu(p[:30, :30], 1) == 0).all()
    np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-14)
    o_r, l_r = oracle.attn_fwd_rows(qb, kb, vb, 0.4, [0, 1, 1], [0, 7, 49], causal=True)
    np.testing.assert_array_equal(o_r, o_c.reshape(2, 50, 16)[[0, 1, 1], [0, 7, 49]])


# ---------------------------------------------------------------- backward

def _autograd_f64(qb, kb, vb, dob, scale, causal):
    q, k, v = (_f64(x).requires_grad_(True) for x in (qb, kb, vb))
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, scale=scale, is_causal=causal)
    o.backward(_f64(dob))
    return q.grad.numpy(), k.grad.numpy(), v.grad.numpy()


@pytest.mark.parametrize("shape,causal", [((1, 2, 48, 64, 32), False), ((2, 1, 40, 24, 16), True),
                                          ((1, 1, 30, 90, 16), True), ((1, 2, 128, 128, 128), False)])
def test_backward_oracle_matches_autograd_f64(shape, causal):
    B, H, Sq, Sk, D = shape
    qb, kb, vb = wl.make_inputs_bits(B, H, Sq, Sk, D, seed=41)
    dob = wl.make_inputs_bits(B, H, Sq, Sq, D, seed=42)[0]
    scale = 1.0 / math.sqrt(D)
    got = oracle.attn_bwd(qb, kb, vb, dob, scale, causal=causal)
    ref = _autograd_f64(qb, kb, vb, dob, scale, causal)
    for g, r in zip(got, ref):
        np.testing.assert_allclose(g, r, rtol=1e-9, atol=1e-12)


def test_backward_oracle_matches_central_differences():
    # dL/dx for L = sum(O * dO) by central differences of the oracle's own forward, on a
    # handful of entries of each input (fp64 forward through a perturbed fp64 copy).
    B, H, Sq, Sk, D = 1, 1, 6, 5, 4
    qb, kb, vb = wl.make_inputs_bits(B, H, Sq, Sk, D, seed=43, qk_std=1.5)
    dob = wl.make_inputs_bits(B, H, Sq, Sq, D, seed=44)[0]
    scale = 0.7
    for causal in (False, True):
        dq, dk, dv = oracle.attn_bwd(qb, kb, vb, dob, scale, causal=causal)
        q, k, v, do = (online.bf16_bits_to_f64(x)[0, 0] for x in (qb, kb, vb, dob))

        def loss(q_, k_, v_):
            s = scale * q_ @ k_.T
            if causal:
                s = np.where(np.tril(np.ones((Sq, Sk), bool)), s, -np.inf)
            p = np.exp(s - s.max(axis=1, keepdims=True))
            p /= p.sum(axis=1, keepdims=True)
            return float(((p @ v_) * do).sum())

        h = 1e-6
        for which, grad in (("q", dq), ("k", dk), ("v", dv)):
            for (r, d) in ((0, 0), (2, 3), (4, 1)):
                args = {"q": q.copy(), "k": k.copy(), "v": v.copy()}
                args[which][r, d] += h
                lp = loss(args["q"], args["k"], args["v"])
                args[which][r, d] -= 2 * h
                lm = loss(args["q"], args["k"], args["v"])
                assert abs((lp - lm) / (2 * h) - grad[0, 0, r, d]) <= 1e-7, (which, r, d, causal)


def test_backward_closed_forms():
    qb, kb, vb = wl.make_inputs_bits(1, 2, 20, 30, 16, seed=45)
    dob = wl.make_inputs_bits(1, 2, 20, 20, 16, seed=46)[0]
    dq, dk, dv = oracle.attn_bwd(qb, kb, vb, dob, 0.3)
    # sum_j dS_ij = 0 for every row, so dK summed over keys is 0 and dQ is orthogonal to a
    # common shift of all keys; dV summed over keys equals dO summed over queries.
    np.testing.assert_allclose(dk.sum(axis=2), 0.0, atol=1e-12)
    do = online.bf16_bits_to_f64(dob)
    np.testing.assert_allclose(dv.sum(axis=2), do.sum(axis=2), rtol=1e-12, atol=1e-12)
    # zero upstream gradient gives zero gradients
    z = np.zeros_like(dob)
    for g in oracle.attn_bwd(qb, kb, vb, z, 0.3):
        assert not g.any()
