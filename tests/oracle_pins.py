"""Pins for the FP64 oracle: checks against things other than the oracle
itself (arbitrary-precision brute force on a dense layout, closed forms,
invariances, library routines). Each pin takes the loaded oracle library so
that the mutation test can run the same pins against broken builds of it.

A pin raises AssertionError when it fails.
"""
from __future__ import annotations

import math

import mpmath
import numpy as np
import torch

import oracle

BF16, FP16 = oracle.BF16, oracle.FP16
TORCH_DT = {BF16: torch.bfloat16, FP16: torch.float16}


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------------------
# a tiny problem built from a DENSE layout, then scattered into pages
# ---------------------------------------------------------------------------

class Dense:
    """Dense per-sequence K/V plus a paged copy of them.

    The dense tensors are the ground truth; the paged cache is produced by
    scattering them through a random block table (the writer's view), with
    every slot nobody owns filled with NaN, so reading outside the contract
    (past L, or an unused table entry) poisons the result.
    """

    def __init__(self, seed, B, Hq, Hkv, D, bs, lens, dtype=BF16, spare_blocks=5,
                 q=None, k=None, v=None):
        g = torch.Generator().manual_seed(seed)
        rng = np.random.default_rng(seed)
        dt = TORCH_DT[dtype]
        Lmax = max(lens) if lens else 1
        self.B, self.Hq, self.Hkv, self.D, self.bs = B, Hq, Hkv, D, bs
        self.lens = np.asarray(lens, dtype=np.int32)
        self.dtype = dtype
        self.q = q if q is not None else torch.randn(B, Hq, D, generator=g).to(dt)
        self.k = k if k is not None else torch.randn(B, Lmax, Hkv, D, generator=g).to(dt)
        self.v = v if v is not None else torch.randn(B, Lmax, Hkv, D, generator=g).to(dt)
        pages = [(int(L) + bs - 1) // bs for L in lens]
        self.max_blocks = max(1, max(pages) if pages else 1) + 1
        nb = sum(pages) + spare_blocks
        perm = rng.permutation(nb)
        nan = torch.tensor(float("nan")).to(dt)
        kc = torch.full((nb, bs, Hkv, D), nan.item(), dtype=dt)
        vc = torch.full((nb, bs, Hkv, D), nan.item(), dtype=dt)
        table = np.zeros((B, self.max_blocks), dtype=np.int32)
        spare = perm[sum(pages):]
        pos = 0
        for b in range(B):
            for p in range(pages[b]):
                blk = int(perm[pos])
                pos += 1
                table[b, p] = blk
                t0, t1 = p * bs, min(int(lens[b]), (p + 1) * bs)
                kc[blk, : t1 - t0] = self.k[b, t0:t1]
                vc[blk, : t1 - t0] = self.v[b, t0:t1]
            # unused entries point at NaN-filled spare blocks
            for p in range(pages[b], self.max_blocks):
                table[b, p] = int(spare[(b + p) % len(spare)]) if len(spare) else 0
        self.k_cache, self.v_cache, self.table = kc, vc, table
        self.num_blocks = nb
        self.scale = 1.0 / math.sqrt(D)

    def args(self):
        return (_bits(self.q), _bits(self.k_cache), _bits(self.v_cache), self.table,
                self.lens)

    def run(self, lib, scale=None):
        return oracle.paged_decode(*self.args(), self.dtype, self.scale if scale is None else scale,
                                   threads=2, lib=lib)


def brute_force(dense: Dense, scale: float, dps: int = 40) -> np.ndarray:
    """Softmax attention on the dense tensors in mpmath at ``dps`` digits.
    The exponentials are normalised by their plain sum (no max shift), and
    each query head hq reads the dense KV head hq // (Hq / Hkv)."""
    mpmath.mp.dps = dps
    G = dense.Hq // dense.Hkv
    q = dense.q.double().numpy()
    k = dense.k.double().numpy()
    v = dense.v.double().numpy()
    out = np.zeros((dense.B, dense.Hq, dense.D))
    for b in range(dense.B):
        L = int(dense.lens[b])
        for hq in range(dense.Hq):
            if L == 0:
                continue
            h = hq // G
            logits = [mpmath.mpf(scale) * mpmath.fsum(mpmath.mpf(float(x)) * mpmath.mpf(float(y))
                                                      for x, y in zip(q[b, hq], k[b, t, h]))
                      for t in range(L)]
            w = [mpmath.exp(s) for s in logits]
            Z = mpmath.fsum(w)
            for d in range(dense.D):
                out[b, hq, d] = float(mpmath.fsum(w[t] * mpmath.mpf(float(v[b, t, h, d]))
                                                  for t in range(L)) / Z)
    return out


# ---------------------------------------------------------------------------
# pins
# ---------------------------------------------------------------------------

def pin_brute_force(lib):
    """Oracle == arbitrary-precision dense attention on tiny ragged inputs
    (GQA, MQA and MHA geometries, both dtypes, both block sizes)."""
    cases = [
        (1, 2, 8, 2, 8, 4, [1, 5], BF16),
        (2, 3, 4, 2, 8, 4, [9, 16, 3], BF16),
        (3, 2, 6, 1, 4, 8, [17, 8], FP16),
        (4, 2, 2, 2, 8, 16, [33, 2], BF16),
    ]
    for seed, B, Hq, Hkv, D, bs, lens, dt in cases:
        dn = Dense(seed, B, Hq, Hkv, D, bs, lens, dtype=dt)
        got = dn.run(lib)
        ref = brute_force(dn, dn.scale)
        err = np.max(np.abs(got - ref))
        assert np.isfinite(got).all(), "oracle read a slot outside the contract"
        assert err < 1e-12, f"brute force mismatch {err} (case seed {seed})"


def pin_closed_forms(lib):
    """Closed forms: one token returns v_0 exactly; constant V returns V;
    zero query returns the mean of V (numpy.mean); two tokens follow the
    logistic form v0 + sigmoid(s1 - s0) (v1 - v0); one logit 4096 above the
    rest returns that token's v exactly."""
    # one token
    dn = Dense(11, 2, 4, 2, 8, 4, [1, 1])
    got = dn.run(lib)
    G = 2
    for b in range(2):
        for hq in range(4):
            np.testing.assert_array_equal(got[b, hq], dn.v[b, 0, hq // G].double().numpy())
    # constant V across tokens
    dn = Dense(12, 1, 4, 2, 8, 4, [13])
    dn.v[:] = dn.v[:, :1]
    dn = Dense(12, 1, 4, 2, 8, 4, [13], q=dn.q, k=dn.k, v=dn.v)
    got = dn.run(lib)
    for hq in range(4):
        ref = dn.v[0, 0, hq // 2].double().numpy()
        assert np.max(np.abs(got[0, hq] - ref)) < 1e-13, "constant V"
    # zero query: uniform weights, mean of V over the context
    dn = Dense(13, 2, 4, 2, 8, 4, [7, 10])
    dn.q.zero_()
    got = dn.run(lib)
    for b in range(2):
        L = int(dn.lens[b])
        for hq in range(4):
            ref = np.mean(dn.v[b, :L, hq // 2].double().numpy(), axis=0)
            assert np.max(np.abs(got[b, hq] - ref)) < 1e-13, "zero query != mean(V)"
    # two tokens, exact integer logits: q = (2, 1, 0, ...), k0 = (1, 0, ..), k1 = (0, 3, ..)
    # scale 0.5 -> s0 = 1, s1 = 1.5
    D = 8
    q = torch.zeros(1, 1, D)
    q[0, 0, :2] = torch.tensor([2.0, 1.0])
    k = torch.zeros(1, 2, 1, D)
    k[0, 0, 0, 0] = 1.0
    k[0, 1, 0, 1] = 3.0
    v = torch.randn(1, 2, 1, D, generator=torch.Generator().manual_seed(5))
    dn = Dense(14, 1, 1, 1, D, 4, [2], q=q.bfloat16(), k=k.bfloat16(), v=v.bfloat16())
    got = dn.run(lib, scale=0.5)
    sig = 1.0 / (1.0 + math.exp(-(1.5 - 1.0)))
    v0 = dn.v[0, 0, 0].double().numpy()
    v1 = dn.v[0, 1, 0].double().numpy()
    ref = v0 + sig * (v1 - v0)
    assert np.max(np.abs(got[0, 0] - ref)) < 1e-14, "two-token logistic form"
    # one dominant logit
    q = torch.zeros(1, 2, D)
    q[0, :, 0] = 64.0
    k = torch.zeros(1, 9, 1, D)
    k[0, 6, 0, 0] = 64.0
    v = torch.randn(1, 9, 1, D, generator=torch.Generator().manual_seed(6))
    dn = Dense(15, 1, 2, 1, D, 4, [9], q=q.bfloat16(), k=k.bfloat16(), v=v.bfloat16())
    got = dn.run(lib, scale=1.0)
    for hq in range(2):
        np.testing.assert_array_equal(got[0, hq], dn.v[0, 6, 0].double().numpy())


def pin_block_table_invariance(lib):
    """Relabelling physical blocks (cache rows permuted, table remapped) and
    re-paging the same logical K/V with another block size leave the FP64
    result bit-identical."""
    dn = Dense(21, 3, 8, 2, 16, 4, [13, 4, 9])
    base = dn.run(lib)
    rng = np.random.default_rng(3)
    perm = rng.permutation(dn.num_blocks)
    inv = np.empty_like(perm)
    inv[perm] = np.arange(len(perm))
    kc = dn.k_cache.clone()
    vc = dn.v_cache.clone()
    kc[torch.from_numpy(perm)] = dn.k_cache
    vc[torch.from_numpy(perm)] = dn.v_cache
    table = perm[dn.table].astype(np.int32)
    got = oracle.paged_decode(_bits(dn.q), _bits(kc), _bits(vc), table, dn.lens, BF16, dn.scale,
                              threads=2, lib=lib)
    np.testing.assert_array_equal(got, base)
    for bs in (1, 2, 8, 16):
        dn2 = Dense(21, 3, 8, 2, 16, bs, [13, 4, 9], q=dn.q, k=dn.k, v=dn.v)
        np.testing.assert_array_equal(dn2.run(lib), base)


def pin_gqa_reductions(lib):
    """GQA equals MHA over K/V heads repeated G times (torch.repeat_interleave);
    MHA equals independent single-head problems; duplicated query heads in a
    group give identical rows."""
    B, Hq, Hkv, D, bs, lens = 2, 8, 2, 8, 4, [11, 6]
    dn = Dense(31, B, Hq, Hkv, D, bs, lens)
    gqa = dn.run(lib)
    G = Hq // Hkv
    mha = Dense(31, B, Hq, Hq, D, bs, lens, q=dn.q, k=dn.k.repeat_interleave(G, dim=2),
                v=dn.v.repeat_interleave(G, dim=2))
    np.testing.assert_array_equal(mha.run(lib), gqa)
    for hq in range(Hq):
        one = Dense(31, B, 1, 1, D, bs, lens, q=dn.q[:, hq:hq + 1].contiguous(),
                    k=mha.k[:, :, hq:hq + 1].contiguous(), v=mha.v[:, :, hq:hq + 1].contiguous())
        np.testing.assert_array_equal(one.run(lib)[:, 0], gqa[:, hq])
    q = dn.q.clone()
    q[:, 1] = q[:, 0]
    dup = Dense(31, B, Hq, Hkv, D, bs, lens, q=q, k=dn.k, v=dn.v).run(lib)
    np.testing.assert_array_equal(dup[:, 0], dup[:, 1])


def pin_split_merge(lib):
    """Split-K: the LSE merge of the per-split partials equals the unsplit
    result for every split count 1..64; one split is the identity; each
    split's lse equals log(sum exp(s_t)) computed in mpmath."""
    lens = [37, 64, 1, 20]
    dn = Dense(41, 4, 4, 2, 8, 1, lens)  # block size 1: every token its own page
    full = dn.run(lib)
    q, k, v, bt, cl = dn.args()
    for S in range(1, 65):
        chunk = max(1, -(-max(lens) // S))
        lse, o = oracle.split_partials(q, k, v, bt, cl, BF16, dn.scale, chunk, S, lib=lib)
        merged = oracle.lse_merge(lse, o, lib=lib)
        assert np.max(np.abs(merged - full)) < 1e-13, f"split-merge S={S}"
        if S == 1:
            np.testing.assert_array_equal(o[:, :, 0], full)
    # lse of a split against mpmath
    lse, o = oracle.split_partials(q, k, v, bt, cl, BF16, dn.scale, 10, 7, lib=lib)
    mpmath.mp.dps = 40
    qd, kd = dn.q.double().numpy(), dn.k.double().numpy()
    for b, hq, s in [(0, 1, 2), (1, 3, 6), (3, 0, 1), (2, 2, 0), (2, 2, 1)]:
        t0, t1 = s * 10, min(lens[b], (s + 1) * 10)
        if t1 <= t0:
            assert lse[b, hq, s] == -np.inf and not o[b, hq, s].any()
            continue
        ref = mpmath.log(mpmath.fsum(
            mpmath.exp(mpmath.mpf(dn.scale) * mpmath.fsum(
                mpmath.mpf(float(a)) * mpmath.mpf(float(c)) for a, c in zip(qd[b, hq], kd[b, t, hq // 2])))
            for t in range(t0, t1)))
        assert abs(lse[b, hq, s] - float(ref)) < 1e-12, "split lse"


def pin_merge_special_cases(lib):
    """Merge: all-empty rows give zeros; a single non-empty split returns its
    o exactly; two splits with equal lse give the plain average; weights
    follow exp(lse) (a split 1000 below the max contributes nothing)."""
    rng = np.random.default_rng(7)
    o = rng.standard_normal((4, 3, 5))
    lse = np.full((4, 3), -np.inf)
    lse[1, 2] = 3.0
    lse[2, 0] = lse[2, 1] = -1.5
    lse[3, 0], lse[3, 1] = 2.0, -998.0
    out = oracle.lse_merge(lse, o, lib=lib)
    assert not out[0].any()
    np.testing.assert_array_equal(out[1], o[1, 2])
    assert np.max(np.abs(out[2] - 0.5 * (o[2, 0] + o[2, 1]))) < 1e-15
    np.testing.assert_array_equal(out[3], o[3, 0])
    # general weights against mpmath: sum_s e^lse_s o_s / sum_s e^lse_s
    lse = rng.standard_normal((2, 6)) * 30
    o = rng.standard_normal((2, 6, 5))
    out = oracle.lse_merge(lse, o, lib=lib)
    mpmath.mp.dps = 40
    for r in range(2):
        w = [mpmath.exp(mpmath.mpf(float(x))) for x in lse[r]]
        Z = mpmath.fsum(w)
        for d in range(5):
            ref = float(mpmath.fsum(w[s] * mpmath.mpf(float(o[r, s, d])) for s in range(6)) / Z)
            assert abs(out[r, d] - ref) < 1e-13, "merge weights"


def pin_dtype_conversions(lib):
    """Exact decode of all 65536 bf16 and fp16 patterns equals torch's
    upcast; rounding from double equals numpy's float64 -> float16 and
    torch's float32 -> bfloat16 conversions (both round to nearest even),
    and bf16 rounding of a double just above a tie rounds up (no double
    rounding through float32)."""
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    for dt, tdt in ((BF16, torch.bfloat16), (FP16, torch.float16)):
        got = oracle.decode(allbits, dt, lib=lib)
        ref = torch.from_numpy(allbits.view(np.int16)).view(tdt).double().numpy()
        nan = np.isnan(ref)
        assert np.array_equal(np.isnan(got), nan)
        np.testing.assert_array_equal(got[~nan], ref[~nan])
    rng = np.random.default_rng(9)
    x = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-9, 5, 20000),
                        [0.0, -0.0, 65504.0, 65520.0, 70000.0, 6e-8, 3e-8, 2.9e-8]])
    bits16, r16 = oracle.round_to(x, FP16, lib=lib)
    np.testing.assert_array_equal(bits16, x.astype(np.float16).view(np.uint16))
    xf = x.astype(np.float32).astype(np.float64)  # values exactly representable in binary32
    bitsb, rb = oracle.round_to(xf, BF16, lib=lib)
    ref = torch.from_numpy(xf.astype(np.float32)).bfloat16().view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(bitsb, ref)
    # ties and the double-rounding trap
    _, r = oracle.round_to(np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, 1 + 2.0 ** -8 + 2.0 ** -30]),
                           BF16, lib=lib)
    np.testing.assert_array_equal(r, [1.0, 1 + 2.0 ** -6, 1 + 2.0 ** -7])


# ---------------------------------------------------------------------------
# RoPE + paged-KV write
# ---------------------------------------------------------------------------

def _half_ulp(x: np.ndarray, dtype: int) -> np.ndarray:
    """Half a unit in the last place of the storage format at |x| (bf16: 8
    significant bits, fp16: 11 bits with subnormals below 2^-14)."""
    mant, emin = (7, -126) if dtype == BF16 else (10, -14)
    e = np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** emin)))
    return 2.0 ** (e - mant - 1)


class RopeCase:
    """Random q/k/v tokens, a random angle table (any angles: rotation is
    what is pinned, not a frequency schedule), distinct cache slots with one
    padding token (slot -1) and one token whose position is past the table."""

    def __init__(self, seed, dtype, T=7, Hq=4, Hkv=2, D=32, P=9, blocks=5, bs=4):
        g = torch.Generator().manual_seed(seed)
        rng = np.random.default_rng(seed)
        dt = TORCH_DT[dtype]
        self.dtype, self.T, self.Hq, self.Hkv, self.D, self.P = dtype, T, Hq, Hkv, D, P
        self.q = _bits(torch.randn(T, Hq, D, generator=g).to(dt))
        self.k = _bits(torch.randn(T, Hkv, D, generator=g).to(dt))
        self.v = _bits(torch.randn(T, Hkv, D, generator=g).to(dt))
        self.theta = rng.uniform(-4 * np.pi, 4 * np.pi, size=(P, D // 2))
        self.pos = rng.integers(0, P, size=T).astype(np.int32)
        self.pos[-1] = P  # outside the table: the token is skipped
        self.slots = rng.permutation(blocks * bs)[:T].astype(np.int64)
        self.slots[1] = -1  # padding token: q rotated, no cache write
        fill = _bits(torch.full((blocks, bs, Hkv, D), -7.0).to(dt))
        self.kc0, self.vc0 = fill.copy(), fill.copy()
        self.qo0 = _bits(torch.full((T, Hq, D), 5.0).to(dt))

    def table(self, rot_dim):
        th = self.theta[:, : rot_dim // 2]
        return np.concatenate([np.cos(th), np.sin(th)], axis=1).astype(np.float32)

    def run(self, lib, rot_dim, neox, table=None):
        cs = self.table(rot_dim) if table is None else table
        return oracle.rope_kv_write(self.q, self.k, self.v, self.pos, self.slots, cs, rot_dim,
                                    neox, self.dtype, self.kc0, self.vc0, q_out=self.qo0,
                                    lib=lib) + (cs,)


def _complex_rotation(x_bits, cs_row, rot_dim, neox, dtype):
    """Rotation of one head vector written as complex multiplication: pair
    (a, b) is the number x_a + i x_b, turned by e^{i theta_j} (theta_j from
    the table's cos/sin halves). Returns the exact rotated values (float64,
    products of a 16-bit and a 32-bit float are exact in double)."""
    x = oracle.decode(x_bits, dtype)
    half = rot_dim // 2
    a = np.arange(half) if neox else 2 * np.arange(half)
    b = a + half if neox else a + 1
    z = x[..., a] + 1j * x[..., b]
    w = z * (cs_row[:half].astype(np.float64) + 1j * cs_row[half:].astype(np.float64))
    y = x.copy()
    y[..., a], y[..., b] = w.real, w.imag
    return y


def pin_rope_complex_form(lib):
    """Every rotated element is the correctly rounded (within half an ulp)
    value of the complex-multiplication form of the rotary embedding, for
    rotate-halves and interleaved pairing, full and partial rotation, bf16
    and fp16; pass-through dims, V and untouched cache rows are bit-exact;
    a padding slot writes no cache row; an out-of-table position writes
    nothing at all."""
    for dtype in (BF16, FP16):
        for neox in (True, False):
            for rot_dim in (32, 16):
                c = RopeCase(11 + dtype + 2 * neox, dtype)
                q_out, kc, vc, cs = c.run(lib, rot_dim, neox)
                written = np.zeros(kc.shape[0] * kc.shape[1], dtype=bool)
                kcf, vcf = kc.reshape(-1, c.Hkv, c.D), vc.reshape(-1, c.Hkv, c.D)
                for t in range(c.T):
                    if c.pos[t] >= c.P:
                        np.testing.assert_array_equal(q_out[t], c.qo0[t])
                        continue
                    row = cs[c.pos[t]]
                    yq = _complex_rotation(c.q[t], row, rot_dim, neox, dtype)
                    got = oracle.decode(q_out[t], dtype)
                    assert np.all(np.abs(got - yq) <= _half_ulp(yq, dtype)), "q rotation"
                    np.testing.assert_array_equal(q_out[t][:, rot_dim:], c.q[t][:, rot_dim:])
                    if c.slots[t] < 0:
                        continue
                    sl = c.slots[t]
                    written[sl] = True
                    yk = _complex_rotation(c.k[t], row, rot_dim, neox, dtype)
                    got = oracle.decode(kcf[sl], dtype)
                    assert np.all(np.abs(got - yk) <= _half_ulp(yk, dtype)), "k rotation"
                    np.testing.assert_array_equal(kcf[sl][:, rot_dim:], c.k[t][:, rot_dim:])
                    np.testing.assert_array_equal(vcf[sl], c.v[t])
                f0 = c.kc0.reshape(-1, c.Hkv, c.D)
                np.testing.assert_array_equal(kcf[~written], f0[~written])
                np.testing.assert_array_equal(vcf[~written], f0[~written])
                assert written.sum() == c.T - 2


def pin_rope_exact_turns(lib):
    """Angles whose cos/sin are exactly 0 or +-1 give exact results: a zero
    turn is the identity, a half turn negates, a quarter turn maps the pair
    (x_a, x_b) to (-x_b, x_a) with a = j, b = j + rot_dim/2 (rotate-halves)
    or a = 2j, b = 2j + 1 (interleaved)."""
    c = RopeCase(5, BF16, T=3)
    c.pos[:] = [0, 1, 2]
    c.slots[:] = [0, 1, 2]
    D, half = c.D, c.D // 2
    table = np.zeros((c.P, D), dtype=np.float32)
    table[0, :half] = 1.0                      # 0
    table[1, :half] = -1.0                     # pi
    table[2, half:] = 1.0                      # pi / 2
    for neox in (True, False):
        q_out, kc, _, _ = c.run(lib, D, neox, table=table)
        x = oracle.decode(c.q, BF16)
        y = oracle.decode(q_out, BF16)
        np.testing.assert_array_equal(y[0], x[0])
        np.testing.assert_array_equal(y[1], -x[1])
        a = np.arange(half) if neox else 2 * np.arange(half)
        b = a + half if neox else a + 1
        np.testing.assert_array_equal(y[2][:, a], -x[2][:, b])
        np.testing.assert_array_equal(y[2][:, b], x[2][:, a])
        yk = oracle.decode(kc.reshape(-1, c.Hkv, D)[2], BF16)
        xk = oracle.decode(c.k[2], BF16)
        np.testing.assert_array_equal(yk[:, a], -xk[:, b])


# ---------------------------------------------------------------------------
# FP8 E4M3 KV cache with per-kv-head scales
# ---------------------------------------------------------------------------

def pin_e4m3_decode(lib):
    """All 256 E4M3 codes decode to torch's float8_e4m3fn values (NaN codes
    to NaN), including subnormals (m * 2^-9) and the largest finite 448."""
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.decode_e4m3(codes, lib=lib)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan) and nan.sum() == 2
    np.testing.assert_array_equal(got[~nan], ref[~nan])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x08] == 2.0 ** -6


def pin_fp8_kv_equals_dequantised_bf16(lib):
    """FP8 K/V with per-kv-head scales equals the bf16 oracle on the same
    values converted to bf16 (exact: E4M3 values are bf16 values), with each
    head's K scale folded into the logit scale and its V scale into the
    output: rows of kv head h of out_fp8 = v_scale[h] * out_bf16(scale *
    k_scale[h]). Also a per-tensor case (all scales equal)."""
    rng = np.random.default_rng(17)
    B, Hq, Hkv, D, bs = 3, 8, 4, 16, 4
    G = Hq // Hkv
    lens = [1, 9, 23]
    nb = 20
    kf = (torch.randn(nb, bs, Hkv, D, generator=torch.Generator().manual_seed(3)) * 3)
    vf = (torch.randn(nb, bs, Hkv, D, generator=torch.Generator().manual_seed(4)) * 3)
    k8 = kf.to(torch.float8_e4m3fn)
    v8 = vf.to(torch.float8_e4m3fn)
    kb = _bits(k8.to(torch.float32).to(torch.bfloat16))
    vb = _bits(v8.to(torch.float32).to(torch.bfloat16))
    k8n, v8n = k8.view(torch.uint8).numpy(), v8.view(torch.uint8).numpy()
    q = _bits(torch.randn(B, Hq, D, generator=torch.Generator().manual_seed(5)).bfloat16())
    table = rng.permutation(nb)[: B * 6].reshape(B, 6).astype(np.int32)
    cl = np.array(lens, dtype=np.int32)
    scale = D ** -0.5
    for ks, vs in ((np.array([0.5, 2.0, 0.125, 3.0]), np.array([4.0, 0.25, 1.5, 0.75])),
                   (np.full(Hkv, 0.3), np.full(Hkv, 1.7))):
        got = oracle.paged_decode_kv(q, k8n, v8n, table, cl, BF16, oracle.FP8_E4M3, scale, ks, vs,
                                     lib=lib)
        for h in range(Hkv):
            ref = oracle.paged_decode(q, kb, vb, table, cl, BF16, scale * ks[h], lib=lib)
            rows = slice(h * G, (h + 1) * G)
            np.testing.assert_allclose(got[:, rows], vs[h] * ref[:, rows], rtol=1e-12,
                                       atol=1e-12)
    # no scales = unit scales; bf16 caches through the same entry = paged_decode
    got = oracle.paged_decode_kv(q, k8n, v8n, table, cl, BF16, oracle.FP8_E4M3, scale, lib=lib)
    ref = oracle.paged_decode(q, kb, vb, table, cl, BF16, scale, lib=lib)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)
    got = oracle.paged_decode_kv(q, kb, vb, table, cl, BF16, BF16, scale, lib=lib)
    np.testing.assert_array_equal(got, ref)


# ---------------------------------------------------------------------------
# KV-cache movement
# ---------------------------------------------------------------------------

def _kv_problem(seed):
    d = Dense(seed, B=3, Hq=4, Hkv=2, D=8, bs=4, lens=[5, 12, 1], spare_blocks=9)
    d.kc, d.vc, d.q_bits = _bits(d.k_cache), _bits(d.v_cache), _bits(d.q)
    return d


def pin_gather_matches_attention_addressing(lib):
    """Gathered rows are the tokens attention reads: decode attention over
    the gathered contiguous K/V (as a cache of 1-token blocks with an
    identity table) equals decode attention over the paged cache, bit for
    bit in FP64; the gathered K equals the dense K the pages were built from."""
    d = _kv_problem(31)
    kg, vg = oracle.gather_kv(d.kc, d.vc, d.table, d.lens, lib=lib)
    total = int(d.lens.sum())
    assert kg.shape[0] == total
    off = np.concatenate([[0], np.cumsum(d.lens)[:-1]])
    for b in range(d.B):
        np.testing.assert_array_equal(kg[off[b]:off[b] + d.lens[b]], _bits(d.k[b, : d.lens[b]]))
        np.testing.assert_array_equal(vg[off[b]:off[b] + d.lens[b]], _bits(d.v[b, : d.lens[b]]))
    t1 = np.zeros((d.B, int(d.lens.max())), dtype=np.int32)
    for b in range(d.B):
        t1[b, : d.lens[b]] = off[b] + np.arange(d.lens[b])
    ref = oracle.paged_decode(d.q_bits, d.kc, d.vc, d.table, d.lens, BF16, 0.3, lib=lib)
    got = oracle.paged_decode(d.q_bits, kg.reshape(total, 1, d.Hkv, d.D),
                              vg.reshape(total, 1, d.Hkv, d.D), t1, d.lens, BF16, 0.3, lib=lib)
    np.testing.assert_array_equal(got, ref)


def pin_scatter_then_gather_roundtrip(lib):
    """Rows scattered into the slots a block table names come back unchanged
    from a gather through that table; padding rows (slot -1) write nothing;
    slots nobody names keep their bytes."""
    rng = np.random.default_rng(5)
    nb, bs, Hkv, D = 12, 4, 2, 8
    lens = np.array([6, 9], dtype=np.int32)
    table = rng.permutation(nb)[:6].reshape(2, 3).astype(np.int32)
    slots = np.concatenate([table[b, np.arange(L) // bs] * bs + np.arange(L) % bs
                            for b, L in enumerate(lens)]).astype(np.int64)
    rows = rng.integers(0, 65535, size=(slots.size, Hkv, D)).astype(np.uint16)
    rows_v = rng.integers(0, 65535, size=(slots.size, Hkv, D)).astype(np.uint16)
    pad_rows = np.concatenate([rows, rows[:1] ^ 1])
    pad_v = np.concatenate([rows_v, rows_v[:1] ^ 1])
    pad_slots = np.concatenate([slots, [-1]])
    k0 = rng.integers(0, 65535, size=(nb, bs, Hkv, D)).astype(np.uint16)
    v0 = rng.integers(0, 65535, size=(nb, bs, Hkv, D)).astype(np.uint16)
    k1, v1 = oracle.scatter_kv(pad_rows, pad_v, pad_slots, k0, v0, lib=lib)
    kg, vg = oracle.gather_kv(k1, v1, table, lens, lib=lib)
    np.testing.assert_array_equal(kg, rows)
    np.testing.assert_array_equal(vg, rows_v)
    untouched = np.ones(nb * bs, dtype=bool)
    untouched[slots] = False
    np.testing.assert_array_equal(k1.reshape(nb * bs, Hkv, D)[untouched],
                                  k0.reshape(nb * bs, Hkv, D)[untouched])
    np.testing.assert_array_equal(v1.reshape(nb * bs, Hkv, D)[untouched],
                                  v0.reshape(nb * bs, Hkv, D)[untouched])


def pin_compaction_preserves_attention(lib):
    """Compaction: copy every used block to a free block, remap the table
    through the same old -> new map; attention over the moved cache equals
    attention over the original bit for bit, blocks not written keep their
    bytes, and an empty pair list or remapping through the identity changes
    nothing."""
    d = _kv_problem(41)
    used = sorted({int(x) for b in range(d.B)
                   for x in d.table[b, : (int(d.lens[b]) + d.bs - 1) // d.bs]})
    free = [i for i in range(d.kc.shape[0]) if i not in used]
    assert len(free) >= len(used)
    pairs = np.array([[u, free[i]] for i, u in enumerate(used)], dtype=np.int64)
    k1, v1 = oracle.copy_blocks(d.kc, d.vc, pairs, lib=lib)
    new_id = np.arange(d.kc.shape[0], dtype=np.int32)
    new_id[pairs[:, 0]] = pairs[:, 1]
    t1 = oracle.remap_table(d.table, d.lens, d.bs, new_id, lib=lib)
    ref = oracle.paged_decode(d.q_bits, d.kc, d.vc, d.table, d.lens, BF16, 0.2, lib=lib)
    got = oracle.paged_decode(d.q_bits, k1, v1, t1, d.lens, BF16, 0.2, lib=lib)
    np.testing.assert_array_equal(got, ref)
    written = set(int(x) for x in pairs[:, 1])
    for i in range(d.kc.shape[0]):
        if i not in written:
            np.testing.assert_array_equal(k1[i], d.kc[i])
            np.testing.assert_array_equal(v1[i], d.vc[i])
    k2, v2 = oracle.copy_blocks(d.kc, d.vc, np.zeros((0, 2), dtype=np.int64), lib=lib)
    np.testing.assert_array_equal(k2, d.kc)
    np.testing.assert_array_equal(
        oracle.remap_table(d.table, d.lens, d.bs, np.arange(d.kc.shape[0]), lib=lib), d.table)



# ---------------------------------------------------------------------------
# row selection (the entry points the full-size GPU checks and the CPU
# baseline use)
# ---------------------------------------------------------------------------

def pin_row_selection(lib):
    """Selected rows equal the matching rows of the full output, bit for bit,
    and the brute force: shuffled rows, repeated rows and a single row, through
    paged_decode_rows (bf16 and fp16) and paged_decode_kv(rows=...) (bf16 and
    FP8 caches with per-head scales). B = Hq, so a selection that swapped b and
    hq would still address valid rows and could only be caught by its values."""
    rng = np.random.default_rng(23)
    for seed, dt in ((51, BF16), (52, FP16)):
        dn = Dense(seed, B=8, Hq=8, Hkv=2, D=8, bs=4, lens=[5, 12, 1, 7, 3, 9, 16, 2], dtype=dt)
        full = dn.run(lib)
        every = np.array([(b, h) for b in range(8) for h in range(8)], dtype=np.int32)
        selections = [every[rng.permutation(len(every))],
                      every[rng.integers(0, len(every), size=23)],  # repeats
                      np.array([[6, 3]], dtype=np.int32),
                      np.array([[3, 6], [6, 3], [0, 7], [7, 0]], dtype=np.int32)]
        for rows in selections:
            got = oracle.paged_decode_rows(*dn.args(), dt, dn.scale, rows, threads=3, lib=lib)
            np.testing.assert_array_equal(got, full[rows[:, 0], rows[:, 1]])
            got_kv = oracle.paged_decode_kv(*dn.args(), dt, dt, dn.scale, rows=rows, threads=2,
                                            lib=lib)
            np.testing.assert_array_equal(got_kv, full[rows[:, 0], rows[:, 1]])
        bf = brute_force(dn, dn.scale)
        rows = selections[3]
        got = oracle.paged_decode_rows(*dn.args(), dt, dn.scale, rows, lib=lib)
        assert np.max(np.abs(got - bf[rows[:, 0], rows[:, 1]])) < 1e-12
    # FP8 caches with per-head scales: rows of the full FP8 output
    B, Hq, Hkv, D, bs, nb = 6, 6, 3, 16, 4, 30
    g = torch.Generator().manual_seed(61)
    k8 = (torch.randn(nb, bs, Hkv, D, generator=g) * 3).to(torch.float8_e4m3fn)
    v8 = (torch.randn(nb, bs, Hkv, D, generator=g) * 3).to(torch.float8_e4m3fn)
    q = _bits(torch.randn(B, Hq, D, generator=g).bfloat16())
    table = rng.permutation(nb)[: B * 5].reshape(B, 5).astype(np.int32)
    cl = np.array([20, 1, 7, 13, 4, 17], dtype=np.int32)
    ks, vs = np.array([0.5, 2.0, 0.25]), np.array([1.5, 0.75, 3.0])
    k8n, v8n = k8.view(torch.uint8).numpy(), v8.view(torch.uint8).numpy()
    full = oracle.paged_decode_kv(q, k8n, v8n, table, cl, BF16, oracle.FP8_E4M3, 0.25, ks, vs,
                                  lib=lib)
    every = np.array([(b, h) for b in range(B) for h in range(Hq)], dtype=np.int32)
    for rows in (every[rng.permutation(len(every))], every[rng.integers(0, len(every), 9)],
                 np.array([[4, 1]], dtype=np.int32)):
        got = oracle.paged_decode_kv(q, k8n, v8n, table, cl, BF16, oracle.FP8_E4M3, 0.25, ks, vs,
                                     rows=rows, threads=4, lib=lib)
        np.testing.assert_array_equal(got, full[rows[:, 0], rows[:, 1]])


ALL_PINS = [pin_brute_force, pin_closed_forms, pin_block_table_invariance, pin_gqa_reductions,
            pin_split_merge, pin_merge_special_cases, pin_dtype_conversions,
            pin_rope_complex_form, pin_rope_exact_turns, pin_e4m3_decode,
            pin_fp8_kv_equals_dequantised_bf16, pin_gather_matches_attention_addressing,
            pin_scatter_then_gather_roundtrip, pin_compaction_preserves_attention,
            pin_row_selection]
