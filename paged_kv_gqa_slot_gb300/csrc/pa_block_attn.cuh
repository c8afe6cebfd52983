// pa_block_attn.cuh -- the paged-KV pipeline shared by the decode, split-KV and
// warp-MMA prefill kernels.
//
// Producer: one warp walks a sequence's block table (32 entries per coalesced load,
// the next 32 prefetched) and, for each logical block, has two lanes issue the TMA loads
// of the (block, kv head) K tile and V tile into a ring slot of shared memory.  Each tile
// is [16 tokens x D] bf16 = one contiguous 2 or 4 KB run of the pool, loaded as ONE box
// through a 4-D map whose 64-column halves are a dimension of their own (stride 128 B),
// so it lands half-major ([half][16 rows][128 B], 128-byte swizzled).  Per-box cost, not
// bytes, limits a TMA stream of small boxes, so one box per tile rather than one per half
// doubles the rate an SM can pull paged blocks.  The block id is only a coordinate of the
// tensor map, so paging costs nothing beyond the table read.
//
// Consumer: a warp owns a 16-row tile of (query, head) rows.  Per 16-token block it
// computes S = Q K^T with mma.m16n8k16 (Q fragments stay in registers), masks, updates
// the running max / sum (online softmax in base 2, fp32), splits P into high and low bf16
// parts and accumulates O += P V with the same MMA, once on each part, reading K and V with
// ldmatrix (V transposed): O keeps about 16 bits of each weight.  The running sum adds
// hi + lo, the very weights the products use.  The decode form (block_step_heads, below)
// does the same (its multi-query use keeps one part where every row sees many keys at the
// usual scale).
#pragma once

#include "pa_device.cuh"

namespace pa {

template <int D>
struct KvTile {
    static constexpr int kHalves = D / 64;                 // 64-column (128-byte) TMA boxes per tile
    static constexpr int kBoxBytes = kBlockSize * 128;     // 2048
    static constexpr int kTileBytes = kBlockSize * D * 2;  // one (block, kv head) tile of K or of V
    static constexpr int kStageBytes = 2 * kTileBytes;     // K tile then V tile
};

// Issue the TMA loads of logical blocks [blk0, blk0 + n) of one sequence into a ring of
// `stages` slots.  Called by a whole warp; returns false if a wait timed out.  On return
// every copy it issued has landed (or the wait for it timed out), so the caller may exit.
template <int D>
// `first`, when `has_first`, is this lane's entry bt[lane] loaded earlier by the caller (valid
// for lane < n), so that the first copies need not wait for that load.
__device__ __forceinline__ bool produce_kv_blocks(uint8_t* ring, int stages, uint64_t* full, uint64_t* empty,
                                                  const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                                                  const int32_t* bt, int n, int num_blocks, int num_kv_heads,
                                                  int kvh, unsigned* status, uint64_t policy, int first = 0,
                                                  bool has_first = false) {
    using T = KvTile<D>;
    const int lane = threadIdx.x & 31;
    int next = (lane < n) ? (has_first ? first : __ldg(bt + lane)) : 0;
    bool ok = true;
    int issued = 0;
    for (int c0 = 0; c0 < n && ok; c0 += 32) {
        int cur = next;
        if (c0 + 32 + lane < n) next = __ldg(bt + c0 + 32 + lane);
        if (c0 + lane < n && (cur < 0 || cur >= num_blocks)) {
            atomicOr(status, kDevOutOfRange);
            cur = 0;  // keep the copy inside the pool; the status word reports the bad id
        }
        const int cnt = min(32, n - c0);
        for (int j = 0; j < cnt; ++j) {
            const int blk = __shfl_sync(0xffffffffu, cur, j);
            const int i = c0 + j;
            const int st = i % stages;
            if (lane == 0) {
                if (i >= stages) ok = mbar_wait(&empty[st], ((i / stages) & 1) ^ 1);
                if (ok) mbar_arrive_expect_tx(&full[st], T::kStageBytes);
            }
            ok = __shfl_sync(0xffffffffu, ok, 0) != 0;
            if (!ok) break;
            // the K and V boxes of the block go out from lanes 0 and 1 in one instruction
            if (lane < 2)
                tma_load_tile(ring + st * T::kStageBytes + lane * T::kTileBytes, lane == 0 ? tm_k : tm_v,
                              blk * num_kv_heads + kvh, &full[st], policy);
            ++issued;
        }
    }
    // every copy this warp issued must have landed before the CTA may leave
    if (lane == 0) {
        for (int i = max(0, issued - stages); i < issued; ++i)
            if (!mbar_wait(&full[i % stages], (i / stages) & 1)) ok = false;
        if (!ok) atomicOr(status, kDevTimeout);
    }
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Running softmax state of the two rows a thread touches (row lane/4 and lane/4 + 8).
struct RowState {
    float m_a, l_a, m_b, l_b;
    __device__ __forceinline__ void init() {
        m_a = -INFINITY;
        l_a = 0.f;
        m_b = -INFINITY;
        l_b = 0.f;
    }
};

// Fragments of a warp's 16-row tile.  With TWO_ROWS the tile uses all 16 MMA rows
// (lane/4 and lane/4 + 8); without it only rows 0..7 carry data (a group of <= 8 query
// heads) and the A/C registers of rows 8..15 are never materialised: the MMA reads zero
// for them and its row 8..15 outputs are dead values.
template <bool TWO_ROWS>
struct Rows {
    static constexpr int kA = TWO_ROWS ? 4 : 2;  // A registers per 16-wide k step
    static constexpr int kC = TWO_ROWS ? 4 : 2;  // C registers per 8-wide n tile
};

// c[16x8] += a[16x16] * b[16x8] (bf16 in, fp32 accumulate) on the tile's live rows.
template <bool TWO_ROWS>
__device__ __forceinline__ void mma_rows(float (&c)[Rows<TWO_ROWS>::kC], const uint32_t (&a)[Rows<TWO_ROWS>::kA],
                                         uint32_t b0, uint32_t b1) {
    if constexpr (TWO_ROWS) {
        asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
            "{%0, %1, %2, %3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
    } else {
        float d2, d3;
        asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %6, %5, %6}, {%7, %8}, "
            "{%0, %1, %9, %9};"
            : "+f"(c[0]), "+f"(c[1]), "=f"(d2), "=f"(d3)
            : "r"(a[0]), "r"(a[1]), "r"(0u), "r"(b0), "r"(b1), "f"(0.f));
    }
}

// Online-softmax update of one row from its four scores in this thread (keys t0, t0+1,
// t0+8, t0+9 of the block); returns P's two packed bf16 pairs, as high parts (p01, p89) and
// low parts (q01, q89: bf16(p - hi)), and alpha.  The running sum adds hi + lo, the weights
// the two P V products apply.
struct RowUpdate {
    uint32_t p01, p89, q01, q89;
    float alpha;
};
__device__ __forceinline__ RowUpdate row_update(float& m, float& l, float s0, float s1, float s8, float s9, int t0,
                                                int lim, float scale_log2) {
    float x0 = t0 < lim ? s0 * scale_log2 : -INFINITY;
    float x1 = t0 + 1 < lim ? s1 * scale_log2 : -INFINITY;
    float x2 = t0 + 8 < lim ? s8 * scale_log2 : -INFINITY;
    float x3 = t0 + 9 < lim ? s9 * scale_log2 : -INFINITY;
    float mx = fmaxf(fmaxf(x0, x1), fmaxf(x2, x3));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float mn = fmaxf(m, mx);
    const float base = mn == -INFINITY ? 0.f : mn;  // a row that has seen no key yet
    RowUpdate u;
    u.alpha = fast_exp2(m - base);
    const float p0 = fast_exp2(x0 - base), p1 = fast_exp2(x1 - base);
    const float p2 = fast_exp2(x2 - base), p3 = fast_exp2(x3 - base);
    x0 = round_bf16(p0);
    x1 = round_bf16(p1);
    x2 = round_bf16(p2);
    x3 = round_bf16(p3);
    const float y0 = round_bf16(p0 - x0), y1 = round_bf16(p1 - x1);
    const float y2 = round_bf16(p2 - x2), y3 = round_bf16(p3 - x3);
    l = l * u.alpha + (((x0 + y0) + (x1 + y1)) + ((x2 + y2) + (x3 + y3)));
    m = mn;
    u.p01 = pack_bf16x2(x0, x1);
    u.p89 = pack_bf16x2(x2, x3);
    u.q01 = pack_bf16x2(y0, y1);
    u.q89 = pack_bf16x2(y2, y3);
    return u;
}

// One 16-token block for one warp's 16-row tile.
//   ks, vs   : shared addresses of the K and V tiles of the ring slot
//   qa       : Q A-fragments of the warp's rows, [D/16][kA]
//   o        : O accumulators, [D/8][kC] (C-fragment layout)
//   lim_a/b  : keys with in-block index < lim are visible to row a (lane/4) / row b
//              (lane/4 + 8); <= 0 means none
//   vlim     : rows >= vlim of the slot lie past the sequence end; whatever they hold
//              (stale data, even NaN) is zeroed in the V fragments, since P = 0 times
//              NaN would still poison O.  K needs no such care: masked scores are
//              replaced, not scaled.
template <int D, bool TWO_ROWS>
__device__ __forceinline__ void block_step(uint32_t ks, uint32_t vs,
                                           const uint32_t (&qa)[D / 16][Rows<TWO_ROWS>::kA],
                                           float (&o)[D / 8][Rows<TWO_ROWS>::kC], RowState& rs, int lim_a,
                                           int lim_b, int vlim, float scale_log2) {
    constexpr int kC = Rows<TWO_ROWS>::kC;
    const int lane = threadIdx.x & 31;
    float s0[kC], s1[kC];
#pragma unroll
    for (int j = 0; j < kC; ++j) s0[j] = s1[j] = 0.f;
    {
        const int mi = lane >> 3, rr = lane & 7;
        const int tok = rr + ((mi >> 1) << 3);  // matrices 0,1: tokens 0-7; 2,3: tokens 8-15
        const int csel = mi & 1;                // matrices 0,2: first 8 columns of the k-step
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const int chunk = kk * 2 + csel;
            const uint32_t addr = ks + (chunk >> 3) * KvTile<D>::kBoxBytes + swz128(tok, chunk & 7);
            uint32_t b0, b1, b2, b3;
            ldsm_x4(addr, b0, b1, b2, b3);
            mma_rows<TWO_ROWS>(s0, qa[kk], b0, b1);
            mma_rows<TWO_ROWS>(s1, qa[kk], b2, b3);
        }
    }
    const int t0 = (lane & 3) * 2;  // this thread's key columns: t0, t0+1, t0+8, t0+9
    uint32_t pa[Rows<TWO_ROWS>::kA], pl[Rows<TWO_ROWS>::kA];  // P's high and low parts
    {
        const RowUpdate u = row_update(rs.m_a, rs.l_a, s0[0], s0[1], s1[0], s1[1], t0, lim_a, scale_log2);
#pragma unroll
        for (int j = 0; j < D / 8; ++j) {
            o[j][0] *= u.alpha;
            o[j][1] *= u.alpha;
        }
        if constexpr (TWO_ROWS) {
            pa[0] = u.p01;
            pa[2] = u.p89;
            pl[0] = u.q01;
            pl[2] = u.q89;
        } else {
            pa[0] = u.p01;
            pa[1] = u.p89;
            pl[0] = u.q01;
            pl[1] = u.q89;
        }
    }
    if constexpr (TWO_ROWS) {
        const RowUpdate u = row_update(rs.m_b, rs.l_b, s0[2], s0[3], s1[2], s1[3], t0, lim_b, scale_log2);
#pragma unroll
        for (int j = 0; j < D / 8; ++j) {
            o[j][2] *= u.alpha;
            o[j][3] *= u.alpha;
        }
        pa[1] = u.p01;
        pa[3] = u.p89;
        pl[1] = u.q01;
        pl[3] = u.q89;
    }
    {
        const int mi = lane >> 3, rr = lane & 7;
        const int tok = rr + ((mi & 1) << 3);  // matrices 0,2: tokens 0-7; 1,3: tokens 8-15
        const int csel = mi >> 1;              // matrices 0,1: even 8-column chunk; 2,3: odd
        // transposed fragments: b0/b2 hold keys t0 (low half) and t0+1 (high half), b1/b3
        // keys t0+8 and t0+9; keys at or past vlim are zeroed
        const uint32_t m0 = vlim >= kBlockSize ? 0xffffffffu
                                               : (t0 < vlim ? 0x0000ffffu : 0u) | (t0 + 1 < vlim ? 0xffff0000u : 0u);
        const uint32_t m1 = vlim >= kBlockSize ? 0xffffffffu
                                               : (t0 + 8 < vlim ? 0x0000ffffu : 0u) | (t0 + 9 < vlim ? 0xffff0000u : 0u);
#pragma unroll
        for (int nn = 0; nn < D / 16; ++nn) {
            const int chunk = nn * 2 + csel;
            const uint32_t addr = vs + (chunk >> 3) * KvTile<D>::kBoxBytes + swz128(tok, chunk & 7);
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(addr, b0, b1, b2, b3);
            mma_rows<TWO_ROWS>(o[2 * nn], pa, b0 & m0, b1 & m1);
            mma_rows<TWO_ROWS>(o[2 * nn + 1], pa, b2 & m0, b3 & m1);
            mma_rows<TWO_ROWS>(o[2 * nn], pl, b0 & m0, b1 & m1);
            mma_rows<TWO_ROWS>(o[2 * nn + 1], pl, b2 & m0, b3 & m1);
        }
    }
}

// Q A-fragments of a 16-row tile from global memory.  row_a / row_b: the rows this
// thread feeds (lane/4 and lane/4 + 8), nullptr for a padding row.
template <int D, bool TWO_ROWS>
__device__ __forceinline__ void load_q_frags(uint32_t (&qa)[D / 16][Rows<TWO_ROWS>::kA], const __nv_bfloat16* row_a,
                                             const __nv_bfloat16* row_b) {
    const int c = (threadIdx.x & 3) * 2;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t lo = row_a ? ld_u32(row_a + kk * 16 + c) : 0u;
        const uint32_t hi = row_a ? ld_u32(row_a + kk * 16 + c + 8) : 0u;
        if constexpr (TWO_ROWS) {
            qa[kk][0] = lo;
            qa[kk][2] = hi;
            qa[kk][1] = row_b ? ld_u32(row_b + kk * 16 + c) : 0u;
            qa[kk][3] = row_b ? ld_u32(row_b + kk * 16 + c + 8) : 0u;
        } else {
            qa[kk][0] = lo;
            qa[kk][1] = hi;
        }
    }
}

// ------------------------------------------------------------------------------------
// Decode form: the query heads of one kv group are the MMA's N dimension (8 per n-tile),
// the block's 16 tokens (for S^T = K Q^T) and head_dim (for O^T = V^T P^T) are its M
// dimension, so a block costs 2 * D/16 MMAs per 8 heads with no padding rows.  Each
// thread holds, per n-tile, heads nt*8 + 2*(lane%4) (+1) for tokens lane/4 and lane/4+8.
// The P^T accumulator fragment becomes the B operand of the P V product through two
// in-register 8x8 transposes (movmatrix).

// Per-thread softmax state of its two heads (hA = 2*(lane%4), hB = hA + 1) per n-tile.
template <int NT>
struct HeadState {
    float m[NT][2], l[NT][2];
    __device__ __forceinline__ void init() {
#pragma unroll
        for (int t = 0; t < NT; ++t) m[t][0] = m[t][1] = -INFINITY, l[t][0] = l[t][1] = 0.f;
    }
};

// Q as B fragments: qb[nt][kk] = {Q[h][kk*16 + 2t], +1}, {Q[h][kk*16 + 8 + 2t], +1} with
// h = nt*8 + lane/4; rows >= g (nullptr) are zero.
template <int D, int NT>
__device__ __forceinline__ void load_q_heads(uint32_t (&qb)[NT][D / 16][2], const __nv_bfloat16* qg, int g) {
    const int lane = threadIdx.x & 31, c = (lane & 3) * 2;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int h = nt * 8 + (lane >> 2);
        const __nv_bfloat16* row = h < g ? qg + (size_t)h * D : nullptr;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            qb[nt][kk][0] = row ? ld_u32(row + kk * 16 + c) : 0u;
            qb[nt][kk][1] = row ? ld_u32(row + kk * 16 + c + 8) : 0u;
        }
    }
}

// Multi-query form: column n is (query n / g, head n % g) of a chunk of C queries starting at
// token q0 of the q tensor (rows >= C * g are zero).
template <int D, int NT>
__device__ __forceinline__ void load_q_rows(uint32_t (&qb)[NT][D / 16][2], const __nv_bfloat16* q, int q0, int C,
                                            int g, int num_heads, int kvh) {
    const int lane = threadIdx.x & 31, c = (lane & 3) * 2;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int n = nt * 8 + (lane >> 2);
        const __nv_bfloat16* row =
            n < C * g ? q + ((size_t)(q0 + n / g) * num_heads + (size_t)kvh * g + n % g) * D : nullptr;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            qb[nt][kk][0] = row ? ld_u32(row + kk * 16 + c) : 0u;
            qb[nt][kk][1] = row ? ld_u32(row + kk * 16 + c + 8) : 0u;
        }
    }
}

// One head column's update from this thread's two tokens (x0: token lane/4, x8: lane/4+8)
// with P as one bf16 value: returns alpha and writes the two probabilities back into x0, x8,
// rounded to bf16 (the P V operand), which is also what the running sum adds.
__device__ __forceinline__ float head_update_one(float& m, float& l, float& x0, float& x8) {
    float mx = fmaxf(x0, x8);
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
    const float mn = fmaxf(m, mx);
    const float base = mn == -INFINITY ? 0.f : mn;
    const float alpha = fast_exp2(m - base);
    x0 = round_bf16(fast_exp2(x0 - base));
    x8 = round_bf16(fast_exp2(x8 - base));
    l = l * alpha + (x0 + x8);
    m = mn;
    return alpha;
}

// The same update with P in two parts; returns alpha.  Each probability p is carried as two
// bf16 values, hi = bf16(p) in x0, x8
// and lo = bf16(p - hi) in y0, y8 (p - hi is exact in fp32), which the P V product takes as
// two MMAs: together they hold p to about 16 significant bits instead of 8, and the running
// sum adds hi + lo, the weights the product uses.  With one bf16 P the weights of a row that
// few keys dominate are off by up to 2^-9 of themselves, which moves O by up to 2^-9 times
// the spread of those keys' V -- a few 1e-3 at unit-variance V, enough, added to the final
// rounding of O to bf16, to cross a 1e-2 bound.
__device__ __forceinline__ float head_update(float& m, float& l, float& x0, float& x8, float& y0, float& y8) {
    float mx = fmaxf(x0, x8);
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
    const float mn = fmaxf(m, mx);
    const float base = mn == -INFINITY ? 0.f : mn;
    const float alpha = fast_exp2(m - base);
    const float p0 = fast_exp2(x0 - base), p8 = fast_exp2(x8 - base);
    x0 = round_bf16(p0);
    x8 = round_bf16(p8);
    y0 = round_bf16(p0 - x0);
    y8 = round_bf16(p8 - x8);
    l = l * alpha + ((x0 + y0) + (x8 + y8));
    m = mn;
    return alpha;
}

// One 16-token block for all g <= 8*NT heads of a kv group.
//   ot[nt][mt][4]: O^T accumulators, d = mt*16 + lane/4 (+8), head nt*8 + 2*(lane%4) (+1)
//   valid        : keys with in-block index < valid exist (the rest are masked and their
//                  V rows zeroed in the fragments, whatever the slot holds)
// With MQ the columns are the (query, head) rows of a multi-query chunk: column j of this
// thread in n-tile nt sees keys up to absolute position colpos[nt][j] (causal), and the
// block's first key is at kbase.  With TWO, P is carried as high and low bf16 parts
// (head_update) and the P V product runs once on each; without, as one (head_update_one).
template <int D, int NT, bool MQ, bool TWO>
__device__ __forceinline__ void block_step_heads(uint32_t ks, uint32_t vs, const uint32_t (&qb)[NT][D / 16][2],
                                                 float (&ot)[NT][D / 16][4], HeadState<NT>& hs, int valid,
                                                 float scale_log2, const int (*colpos)[2] = nullptr,
                                                 int kbase = 0) {
    const int lane = threadIdx.x & 31;
    const int mi = lane >> 3, rr = lane & 7;
    const int ltok = rr + ((mi & 1) << 3);  // K matrices 0,2: tokens 0-7; 1,3: tokens 8-15
    const int lcs = mi >> 1;                // K matrices 0,1: even d-chunk; 2,3: odd
    float st[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) st[nt][0] = st[nt][1] = st[nt][2] = st[nt][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const int chunk = kk * 2 + lcs;
        uint32_t a0, a1, a2, a3;
        ldsm_x4(ks + (chunk >> 3) * KvTile<D>::kBoxBytes + swz128(ltok, chunk & 7), a0, a1, a2, a3);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_16816(st[nt], a0, a1, a2, a3, qb[nt][kk][0], qb[nt][kk][1]);
    }
    const int t0 = lane >> 2;  // this thread's tokens: t0 and t0 + 8
    const bool v0 = t0 < valid, v8 = t0 + 8 < valid;
    uint32_t pb[NT][2], pl[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        bool va0 = v0, va8 = v8, vb0 = v0, vb8 = v8;
        if (MQ) {
            const int la = colpos[nt][0] - kbase, lb = colpos[nt][1] - kbase;
            va0 = t0 <= la;
            va8 = t0 + 8 <= la;
            vb0 = t0 <= lb;
            vb8 = t0 + 8 <= lb;
        }
        float xa0 = va0 ? st[nt][0] * scale_log2 : -INFINITY, xa8 = va8 ? st[nt][2] * scale_log2 : -INFINITY;
        float xb0 = vb0 ? st[nt][1] * scale_log2 : -INFINITY, xb8 = vb8 ? st[nt][3] * scale_log2 : -INFINITY;
        float ya0 = 0.f, ya8 = 0.f, yb0 = 0.f, yb8 = 0.f;
        const float aa = TWO ? head_update(hs.m[nt][0], hs.l[nt][0], xa0, xa8, ya0, ya8)
                             : head_update_one(hs.m[nt][0], hs.l[nt][0], xa0, xa8);
        const float ab = TWO ? head_update(hs.m[nt][1], hs.l[nt][1], xb0, xb8, yb0, yb8)
                             : head_update_one(hs.m[nt][1], hs.l[nt][1], xb0, xb8);
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
            ot[nt][mt][0] *= aa;
            ot[nt][mt][2] *= aa;
            ot[nt][mt][1] *= ab;
            ot[nt][mt][3] *= ab;
        }
        // P^T rows (tokens) t0 / t0+8, columns (heads) 2t, 2t+1 -> transposed: the B operand
        pb[nt][0] = movmatrix_t(pack_bf16x2(xa0, xb0));
        pb[nt][1] = movmatrix_t(pack_bf16x2(xa8, xb8));
        if (TWO) {
            pl[nt][0] = movmatrix_t(pack_bf16x2(ya0, yb0));
            pl[nt][1] = movmatrix_t(pack_bf16x2(ya8, yb8));
        }
    }
    // V^T A fragments (ldmatrix.trans): matrices 0,1: tokens 0-7, 2,3: tokens 8-15;
    // 0,2: even d-chunk, 1,3: odd.  a0/a1 hold keys 2t, 2t+1; a2/a3 keys 2t+8, 2t+9.
    const int vtok = rr + ((mi >> 1) << 3);
    const int vcs = mi & 1;
    const int tk = (lane & 3) * 2;
    const uint32_t m0 = valid >= kBlockSize ? 0xffffffffu
                                            : (tk < valid ? 0x0000ffffu : 0u) | (tk + 1 < valid ? 0xffff0000u : 0u);
    const uint32_t m8 = valid >= kBlockSize ? 0xffffffffu
                                            : (tk + 8 < valid ? 0x0000ffffu : 0u) | (tk + 9 < valid ? 0xffff0000u : 0u);
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
        const int chunk = mt * 2 + vcs;
        uint32_t a0, a1, a2, a3;
        ldsm_x4_t(vs + (chunk >> 3) * KvTile<D>::kBoxBytes + swz128(vtok, chunk & 7), a0, a1, a2, a3);
        a0 &= m0;
        a1 &= m0;
        a2 &= m8;
        a3 &= m8;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            mma_16816(ot[nt][mt], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
            if (TWO) mma_16816(ot[nt][mt], a0, a1, a2, a3, pl[nt][0], pl[nt][1]);
        }
    }
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
}  // namespace pa
