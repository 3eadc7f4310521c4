"""The decode kernels' tensor-core page step (csrc/pkv_mma.cuh), modelled on the
CPU: host logic of its index arithmetic, no attention arithmetic of the oracle.

A page tile (16 token rows x D dims, bf16) sits in shared memory as the
128-byte-swizzled tiled TMA boxes write it: box j holds dims 64j .. 64j + 63 of
the 16 rows, 128 bytes per row, and the 16-byte chunk cc of row t lands at
chunk position cc XOR (t mod 8). The model then plays the warp's 32 lanes
through the operand layouts the PTX ISA gives for ldmatrix (.x4 and .trans),
movmatrix (.trans) and mma.sync m16n8k16 (row.col, bf16 in, fp32 out), with the
row addresses and fragment registers the kernel computes, and checks that the
products are exactly S^T = K Q^T and O^T = V^T P^T of the page, that no
ldmatrix phase has a bank conflict, and that the tail mask keeps NaN in unused
rows out of the accumulators. Over several pages, the running max, the
warp-wide rescale vote and the sums of the bf16-rounded weights give the
softmax mean within the weights' rounding.
"""
import numpy as np
import pytest

PAGE = 16
LANES = np.arange(32)


def swz(t, c):
    """the kernel's byte offset of 16-byte chunk c of token row t"""
    return (c >> 3) * 2048 + t * 128 + (((c & 7) ^ (t & 7)) << 4)


def tma_tile(x, D):
    """shared-memory bytes of a [16, D] tile as the swizzled boxes write it: element index per 2-byte slot"""
    slots = np.full(PAGE * D, -1, np.int64)  # slot -> flat element index t * D + d
    for j in range(D // 64):
        for t in range(PAGE):
            for cc in range(8):
                base = j * 2048 + t * 128 + ((cc ^ (t % 8)) * 16)
                for e in range(8):
                    slots[(base + 2 * e) // 2] = t * D + 64 * j + 8 * cc + e
    assert (slots >= 0).all() and len(set(slots.tolist())) == PAGE * D
    return x.reshape(-1)[slots]  # values by 2-byte slot


def offsets(D):
    """the kernel's per-lane ldmatrix row addresses (mma_offsets)"""
    mi, mr = LANES >> 3, LANES & 7
    koff = [swz(mr + ((mi & 1) << 3), 2 * ks + (mi >> 1)) for ks in range(D // 16)]
    voff = [swz(mr + ((mi >> 1) << 3), 2 * ks + (mi & 1)) for ks in range(D // 16)]
    return koff, voff


def ldmatrix(mem, addr, trans=False):
    """.x4: lane L addresses row L % 8 of matrix L // 8; register i of lane L holds the pair
    (row L/4, cols 2(L%4), +1) of matrix i, or of its transpose with .trans"""
    regs = np.zeros((4, 32, 2))
    for i in range(4):
        m = np.stack([mem[(addr[8 * i + r]) // 2:(addr[8 * i + r]) // 2 + 8] for r in range(8)])  # 8 x 8
        if trans:
            m = m.T
        for L in range(32):
            regs[i, L] = m[L // 4, 2 * (L % 4):2 * (L % 4) + 2]
    return regs


def movmatrix_t(frag):
    """movmatrix.trans: lane L holds (row L/4, cols 2(L%4), +1) of M before, of M^T after"""
    m = np.zeros((8, 8))
    for L in range(32):
        m[L // 4, 2 * (L % 4):2 * (L % 4) + 2] = frag[L]
    return np.stack([m.T[L // 4, 2 * (L % 4):2 * (L % 4) + 2] for L in range(32)])


def mma(c, a, b0, b1):
    """m16n8k16 row.col: A regs (rows g / g+8, cols 2c.. / 2c+8..), B regs (k 2c.. / 2c+8.., col g),
    C pairs (row g, cols 2c, 2c+1) and (row g+8, ...); g = lane / 4, c = lane % 4"""
    A, B = np.zeros((16, 16)), np.zeros((16, 8))
    for L in range(32):
        g, k = L // 4, 2 * (L % 4)
        A[g, k:k + 2], A[g + 8, k:k + 2], A[g, k + 8:k + 10], A[g + 8, k + 8:k + 10] = a[0, L], a[1, L], a[2, L], a[3, L]
        B[k:k + 2, g], B[k + 8:k + 10, g] = b0[L], b1[L]
    C = A @ B
    out = c.copy()
    for L in range(32):
        g, k = L // 4, 2 * (L % 4)
        out[L] += [C[g, k], C[g, k + 1], C[g + 8, k], C[g + 8, k + 1]]
    return out


def page_step(K, V, q, nv):
    """the kernel's page step with unit scale, one page, no running state: returns S^T [16, 8] (masked)
    and the unnormalised O^T [D, 8] accumulated from p = 2^(s - max)"""
    D = K.shape[1]
    kmem, vmem = tma_tile(K, D), tma_tile(V, D)
    koff, voff = offsets(D)
    g, c = LANES // 4, LANES % 4
    # Q^T as the B operand: head g, dims 16 ks + 2c (+1) and 16 ks + 8 + 2c (+1)
    qf = [(np.stack([q[g, 16 * ks + 2 * c], q[g, 16 * ks + 2 * c + 1]], 1),
           np.stack([q[g, 16 * ks + 8 + 2 * c], q[g, 16 * ks + 9 + 2 * c]], 1)) for ks in range(D // 16)]
    s = np.zeros((32, 4))
    for ks in range(D // 16):
        s = mma(s, ldmatrix(kmem, koff[ks]), *qf[ks])
    valid = np.stack([g < nv, g < nv, g + 8 < nv, g + 8 < nv], 1)
    s = np.where(valid, s, -np.inf)
    st = np.zeros((16, 8))
    for L in range(32):
        st[g[L], 2 * c[L]:2 * c[L] + 2], st[g[L] + 8, 2 * c[L]:2 * c[L] + 2] = s[L, :2], s[L, 2:]
    mx = st.max(0)  # per head (the kernel: three shuffles over the lanes of a column pair)
    p = np.exp2(s - np.stack([mx[2 * c], mx[2 * c + 1], mx[2 * c], mx[2 * c + 1]], 1))
    pb0, pb1 = movmatrix_t(p[:, :2]), movmatrix_t(p[:, 2:])
    lo = np.stack([2 * c < nv, 2 * c + 1 < nv], 1)
    hi = np.stack([2 * c + 8 < nv, 2 * c + 9 < nv], 1)
    o = np.zeros((D // 16, 32, 4))
    for ks in range(D // 16):
        vf = ldmatrix(vmem, voff[ks], trans=True)
        vf = np.stack([np.where(lo, vf[0], 0), np.where(lo, vf[1], 0), np.where(hi, vf[2], 0), np.where(hi, vf[3], 0)])
        o[ks] = mma(o[ks], vf, pb0, pb1)
    ot = np.zeros((D, 8))
    for ks in range(D // 16):
        for L in range(32):
            ot[16 * ks + g[L], 2 * c[L]:2 * c[L] + 2] = o[ks, L, :2]
            ot[16 * ks + g[L] + 8, 2 * c[L]:2 * c[L] + 2] = o[ks, L, 2:]
    return st, ot, mx


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("nv", [16, 11, 1])
def test_page_step_computes_scores_and_values(D, nv):
    rng = np.random.default_rng(D + nv)
    K = rng.integers(-8, 9, (PAGE, D)).astype(np.float64)  # small integers: every product and sum exact
    V = rng.integers(-8, 9, (PAGE, D)).astype(np.float64)
    q = np.zeros((8, D))
    q[:5] = rng.integers(-3, 4, (5, D))  # a group of 5 heads in the 8 columns, the rest zero
    V[nv:] = np.nan  # unused slots may hold anything
    K[nv:] = np.nan
    st, ot, mx = page_step(K, V, q, nv)
    want_s = K[:nv] @ q.T
    assert np.array_equal(st[:nv], want_s) and np.isneginf(st[nv:]).all()
    p = np.exp2(want_s - want_s.max(0))
    assert np.allclose(ot, V[:nv].T @ p, rtol=1e-12, atol=0) and np.isfinite(ot).all()


@pytest.mark.parametrize("D", [64, 128])
def test_ldmatrix_phases_are_conflict_free_and_cover_the_tile(D):
    koff, voff = offsets(D)
    for offs in (koff, voff):
        seen = set()
        for ks, off in enumerate(offs):
            for i in range(4):  # one 8-row phase per matrix: eight distinct 16-byte bank groups
                rows = off[8 * i:8 * i + 8]
                assert len({(a % 128) // 16 for a in rows}) == 8
            for a in off:
                assert a % 16 == 0 and 0 <= a and a + 16 <= PAGE * D * 2
                seen.add(a)
        assert len(seen) == PAGE * D * 2 // 16  # every 16-byte chunk of the tile read once per product


def bf16(x):
    """round float64 values to bf16 (nearest, ties to even) and back"""
    x = np.asarray(x, np.float64)
    b = x.astype(np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) & 0xFFFF0000
    return b.astype(np.uint32).view(np.float32).astype(np.float64)


def run_pages(K, V, q, n_tok):
    """the kernel's loop over a split's pages with its running state per lane: max (m0, m1 of the lane's two
    heads), partial sums (l0, l1), O^T fragments, rescaled only when some lane's max moved; p rounded to bf16
    and the sums taken over the rounded p. Returns O^T / l per head, [D, 8]."""
    D = K.shape[1]
    g, c = LANES // 4, LANES % 4
    m = np.full((32, 2), -np.inf)
    l = np.zeros((32, 2))
    o = np.zeros((D // 16, 32, 4))
    koff, voff = offsets(D)
    qf = [(np.stack([q[g, 16 * ks + 2 * c], q[g, 16 * ks + 2 * c + 1]], 1),
           np.stack([q[g, 16 * ks + 8 + 2 * c], q[g, 16 * ks + 9 + 2 * c]], 1)) for ks in range(D // 16)]
    for p0 in range(0, n_tok, PAGE):
        nv = min(PAGE, n_tok - p0)
        kmem, vmem = tma_tile(K[p0:p0 + PAGE], D), tma_tile(V[p0:p0 + PAGE], D)
        s = np.zeros((32, 4))
        for ks in range(D // 16):
            s = mma(s, ldmatrix(kmem, koff[ks]), *qf[ks])
        valid = np.stack([g < nv, g < nv, g + 8 < nv, g + 8 < nv], 1)
        s = np.where(valid, s, -np.inf)
        x = np.maximum(s[:, :2], s[:, 2:])
        for sh in (4, 8, 16):  # butterfly over the lanes of a column pair
            x = np.maximum(x, x[LANES ^ sh])
        n = np.maximum(m, x)
        p = bf16(np.exp2(s - np.concatenate([n, n], 1)))
        if (n != m).any():  # the warp-wide vote
            al = np.exp2(m - n)
            l *= al
            o *= np.concatenate([al, al], 1)[None]
            m = n
        l += p[:, :2] + p[:, 2:]
        pb0, pb1 = movmatrix_t(p[:, :2]), movmatrix_t(p[:, 2:])
        lo = np.stack([2 * c < nv, 2 * c + 1 < nv], 1)
        hi = np.stack([2 * c + 8 < nv, 2 * c + 9 < nv], 1)
        for ks in range(D // 16):
            vf = ldmatrix(vmem, voff[ks], trans=True)
            vf = np.stack([np.where(lo, vf[0], 0), np.where(lo, vf[1], 0), np.where(hi, vf[2], 0),
                           np.where(hi, vf[3], 0)])
            o[ks] = mma(o[ks], vf, pb0, pb1)
    for sh in (4, 8, 16):
        l = l + l[LANES ^ sh]
    ot = np.zeros((D, 8))
    for ks in range(D // 16):
        for L in range(32):
            ot[16 * ks + g[L], 2 * c[L]:2 * c[L] + 2] = o[ks, L, :2] / l[L]
            ot[16 * ks + g[L] + 8, 2 * c[L]:2 * c[L] + 2] = o[ks, L, 2:] / l[L]
    return ot


@pytest.mark.parametrize("order", ["rising", "falling"])
def test_split_loop_rescales_to_the_softmax_mean(order):
    # scores whose page maximum rises page after page (a rescale on every page) or falls (none after the first)
    rng = np.random.default_rng(7)
    D, n_tok = 64, 5 * PAGE - 3
    K = bf16(rng.standard_normal((5 * PAGE, D)))
    V = bf16(rng.standard_normal((5 * PAGE, D)))
    q = np.zeros((8, D))
    q[:4] = bf16(rng.standard_normal((4, D)) * 0.3)
    ramp = np.repeat(np.arange(5), PAGE)[:, None] * (1.0 if order == "rising" else -1.0)
    K = bf16(K + ramp * np.sign(q[:4].sum(0))[None] * 0.5)  # shifts every head's scores page by page
    K[n_tok:] = np.nan
    V[n_tok:] = np.nan
    got = run_pages(K, V, q, n_tok)
    s = q[:4] @ K[:n_tok].T  # [4 heads, tokens], log2 domain as in the kernel (unit scale)
    w = np.exp2(s - s.max(1, keepdims=True))
    want = (w @ V[:n_tok] / w.sum(1, keepdims=True)).T  # [D, 4]
    assert np.isfinite(got).all()
    # p is rounded to bf16 in the value product and in the sums: relative weight error <= 2^-8
    assert np.abs(got[:, :4] - want).max() <= 2 ** -8 * np.abs(V[:n_tok]).max()
