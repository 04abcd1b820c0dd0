// tern_gemv.cu -- decode / small-batch ternary-g128 product, M = 1..16.
//
//   y[m][n] = sum_g s[n][g] * sum_{k in g} x[m][k] * (q[n][k] - 1)
//
// ("prism-ml/Ternary-Bonsai-27B-mlx-2bit" model card: ternary g128 weights,
// "Weight representation"; codes unpacked and scaled inside the product,
// "CUDA (NVIDIA GPUs)"; decode is the memory-bandwidth-bound phase,
// "Cross-platform throughput".)
//
// Arithmetic.  At 2.125 bits per weight an M = 1 product must retire ~25 G
// weights per ms to keep HBM busy, more than the CUDA cores can afford at the
// two or three ALU operations a scalar unpack-and-add costs.  So the adds run
// on the tensor pipe (mma.sync m16n8k16, f16 in, f32 accumulate) and the unpack
// is ONE logical AND per two weights:
//
//   * a word holds codes j and j + 8 of a 16-weight slice in bits 2j and
//     2j + 16.  `word & (0x00030003 << 2j)` leaves, in each 16-bit half, the
//     bit pattern q << 2j.  Read as fp16 that is exactly q * 2^(2j - 24) for
//     j <= 4 (a subnormal) and q * 2^-14 for j = 5 (the two low exponent
//     bits), i.e. q * 2^(2j - 24) for every j <= 5 and q = 0, 1, 2.  Codes 6,
//     7, 14, 15 take one shift by 12 and reuse the j = 0 and j = 1 masks.  The
//     result is the MMA A-fragment register directly.  An affine pack, whose
//     code 3 is valid (and would read as 4 in the exponent bits), reads codes
//     5, 6, 7 and 13, 14, 15 after a shift by 10 instead, as slots 0, 1, 2:
//     every slot stays a subnormal and every code 0..3 is exact.
//   * the activation is staged as fp16 B fragments, each value pre-multiplied
//     by the power of two 2^(E + 10 - 2j') that undoes its slot's
//     2^(2j' - 24) (j' = j or j - 6; j or j - 5 for an affine pack), with a
//     per-(token, group) exponent E
//     chosen from the group's max |x| so the largest staged value is below
//     2^15.  bf16 values stage exactly (8 significant bits into 11).  One MMA
//     per slot position j accumulates acc = 2^(E - 14) sum_k q_k x_k over 16
//     weights of 16 rows.
//   * the -1 of q - 1: the same eight-MMA chain run once per (token, group)
//     on the all-ones code pattern gives acc1 = 2^(E - 14) sum_k x_k with the
//     very same rounding, and per row and group
//         y += s_g * (2^(14 - E) * acc - 2^(14 - E) * acc1),
//     so a row of zero weights (q = 1 everywhere) gives exactly 0.
//   * an affine pack (w = s q + b per group, all four codes valid) takes the
//     same two chains: y += s_g * 2^(14 - E) * acc + b_g * 2^(14 - E) * acc1,
//     its biases staged in shared memory beside the scales (AFF).
//
// Work split.  K is cut into S = ceil(G / 8) slices of whole groups (balanced
// to within one group), and N into ranges of 16-row tiles; a CTA owns one
// (slice, range) pair, and the CTAs of slice 0 come first in the grid.  Inside
// a CTA the slice's groups are dealt to the 8 warps as segments: every warp
// takes floor(Gs / 8) whole groups over the full range, and each of the Gs mod
// 8 groups left over is cut into eight tile chunks, one per warp.  A warp
// stages one segment's activation into registers and streams its own
// 32-byte column of every tile of the segment (16 rows x 32 B = one 16-byte
// cp.async per lane) through a private shared-memory ring, kDepth units ahead;
// the first kEarly units go out before the programmatic-dependent-launch wait,
// the rest after staging.  Two tiles per step run as two independent MMA
// chains.  Row partials go to shared memory (private per warp
// for M <= 4, shared atomics beyond) and are summed over the CTA's warps.
// With one slice the CTA stores its rows of y.  With several, the slice-0 CTA
// of a range clears the range's rows of y right after the PDL wait and then
// counts itself into the range's flag word; every other CTA of the range, once
// its loop is done (long after the clearing), waits for that count, counts
// itself and adds its row sums into y with global reductions.  The flag
// counts modulo S (atomicInc), so it is back at 0 when the call ends.  The
// order in which the S slice sums meet is not fixed: the last bits of y may
// differ from run to run.
//
// The 1-bit sibling format (w = (2b - 1) s, bit k%32 of word k/32) runs the
// same kernel with BIN set: a unit is 16 rows x 16 bytes, slot s of a word is
// bits s and s + 16 (read as b * 2^(s' - 24)), MMA j takes slots j and j + 8,
// and y = s F (2 acc - acc1).
//
// The rotation-fused call.  For M <= 2 it is one launch (ROT): each CTA
// rebuilds, in fp32 in shared memory, the 1024-wide slice of the rotated
// activation that its K-slice reads, from H_4096 = H_4 (x) H_1024 (natural
// order): the signed sum of the block's four 1024-wide parts picked by row a
// of H_4 (a = the slice's place in its 4096-block), then a 1024-point
// transform.  The warps stage their groups from it exactly as they stage a
// bf16 x, so x' is never rounded to bf16.  Every row range of a slice repeats
// that work, which is cheap for one or two tokens only; for more tokens
// rotate_stage_kernel runs first: it rotates x once, stages it exactly as the
// product would (exponent and scaled fp16 values, in B-fragment order) into
// the workspace, and the product (PRE) loads the fragments as they are.
#include <mutex>
#include <type_traits>

#include "tern_fwht.cuh"
#include "tern_mma.cuh"

namespace tern {
namespace {

constexpr int kGroup = 128;            // weights per scale
constexpr int kWarps = 8;              // warps per CTA
constexpr int kThreads = kWarps * 32;
constexpr int kDepth = 4;              // units (tile x group) in flight per warp (even)
constexpr int kEarly = 4;              // of which issued before the PDL wait, the rest after staging
constexpr int kSlotBytes = 16 * 32;    // one unit: 16 rows x 32 B of codes
constexpr int kBinSlotBytes = 16 * 16; // one unit of the 1-bit layout: 16 rows x 16 B
constexpr int kMaxTiles = 32;          // tiles per range (bounds partials and scales in shared memory)
constexpr int kPrivateMaxM = 4;        // private per-warp partials up to this many tokens
constexpr size_t kSmemPerSm = 228 * 1024;   // shared memory of one SM
constexpr size_t kCtaSmemReserve = 1024;    // taken by the system from each resident CTA

template <int MT> struct GemvCfg;
template <> struct GemvCfg<1> { static constexpr int kCtasPerSm = 3; };
template <> struct GemvCfg<2> { static constexpr int kCtasPerSm = 2; };

struct GemvArgs {
    const void* x;              // bf16 [M][K], or the rotation's staged fragments (PRE)
    const int* xe;              // PRE: the staging exponent E of each (token, group)
    const int8_t* signs;        // ROT: the rotation's sign pattern [K]
    const uint32_t* codes;      // [N][K/16]
    const __half* scales;       // [N][K/128]
    const __half* biases;       // [N][K/128], an affine pack (AFF) only
    float* y;                   // [M][N]
    // a pair call: a second matrix (N2 rows, T2 tiles) read with the same x;
    // ranges [cps1, cps) are its, [0, cps1) the first one's (cps1 = cps otherwise)
    const uint32_t* codes2;
    const __half* scales2;
    float* y2;
    int N2, T2, cps1;
    unsigned* flag;             // [cps] per-range flag words (S > 1), 0 between calls
    int M, N, K, G, T, S, cps, rmax;
    int gpad;                   // scale row pitch in shared memory (halves)
    int boff;                   // AFF: the staged biases' offset from the scales (halves)
    uint32_t off_sc, off_part;  // shared-memory offsets (bytes)
    uint32_t off_rot;           // ROT: the rotated slice, [M][kRotPitch] fp32
};

__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// The chains of one (16-row, 128-weight) unit for one token tile: the even
// slots and the odd slots accumulate in two independent chains of four MMAs,
// added at the end (acc = even + odd), so consecutive MMAs do not wait on one
// another.  The all-ones pass runs the same two chains and the same addition,
// so a row of zero weights still matches it bit for bit.
template <bool Q3 = false>
__device__ __forceinline__ void mma_chain1(float (&acc)[4], const uint32_t (&w)[4], const uint32_t (&b)[16]) {
    float odd[4];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        uint32_t r[4];
        slot_regs<Q3>(j, w[0], w[1], w[2], w[3], r);
        mma16816((j & 1) ? odd : acc, r[0], r[1], r[2], r[3], b[2 * j], b[2 * j + 1], j > 1);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[e] += odd[e];
}

// Two units of the same group at once: 2 x MT x 2 independent MMA chains
// sharing the B fragments, each unit in the chain order of mma_chain1 (so each
// keeps the ones-pass rounding).
template <int MT, bool Q3 = false>
__device__ __forceinline__ void pair_mmas(float (&acc)[2][MT][4], const uint32_t (&w)[2][4],
                                          const uint32_t (&b)[MT][16]) {
    float odd[2][MT][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        uint32_t r[2][4];
#pragma unroll
        for (int q = 0; q < 2; ++q) slot_regs<Q3>(j, w[q][0], w[q][1], w[q][2], w[q][3], r[q]);
#pragma unroll
        for (int q = 0; q < 2; ++q)
#pragma unroll
            for (int nt = 0; nt < MT; ++nt)
                mma16816((j & 1) ? odd[q][nt] : acc[q][nt], r[q][0], r[q][1], r[q][2], r[q][3], b[nt][2 * j],
                         b[nt][2 * j + 1], j > 1);
    }
#pragma unroll
    for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int nt = 0; nt < MT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[q][nt][e] += odd[q][nt][e];
}

// ---- the 1-bit sibling: bit k%32 of a word is weight k, w = (2b - 1) s ----
// Slot s (0..15) of a word as an fp16 pair: bits s and s + 16 read as
// b * 2^(s' - 24), s' = s for s <= 11 (mantissa, or the low exponent bits for
// 10 and 11), s - 12 for the rest (read after a shift by 12).
__device__ __forceinline__ uint32_t bin_slot(uint32_t w, uint32_t w12, int s) {
    return s < 12 ? (w & (0x00010001u << s)) : (w12 & (0x00010001u << (s - 12)));
}
// One unit's chain for one token tile from this lane's two words (rows gid
// and gid + 8, word t of the group): MMA j takes slots j and j + 8.
__device__ __forceinline__ void bin_chain1(float (&acc)[4], uint32_t w0, uint32_t w1, const uint32_t (&b)[16]) {
    const uint32_t u0 = w0 >> 12, u1 = w1 >> 12;
#pragma unroll
    for (int j = 0; j < 8; ++j)
        mma16816(acc, bin_slot(w0, u0, j), bin_slot(w1, u1, j), bin_slot(w0, u0, j + 8), bin_slot(w1, u1, j + 8),
                 b[2 * j], b[2 * j + 1], j > 0);
}
template <int MT>
__device__ __forceinline__ void bin_pair_mmas(float (&acc)[2][MT][4], const uint32_t (&w)[2][2],
                                              const uint32_t (&b)[MT][16]) {
    uint32_t u[2][2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        u[q][0] = w[q][0] >> 12;
        u[q][1] = w[q][1] >> 12;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int q = 0; q < 2; ++q)
#pragma unroll
            for (int nt = 0; nt < MT; ++nt)
                mma16816(acc[q][nt], bin_slot(w[q][0], u[q][0], j), bin_slot(w[q][1], u[q][1], j),
                         bin_slot(w[q][0], u[q][0], j + 8), bin_slot(w[q][1], u[q][1], j + 8), b[nt][2 * j],
                         b[nt][2 * j + 1], j > 0);
}
// the exact power of two 2^(E + 10 - s') for slot s of the 1-bit layout
__device__ __forceinline__ float bin_stage_multiplier(int E, int s) {
    return __uint_as_float((uint32_t)(E + 10 - (s < 12 ? s : s - 12) + 127) << 23);
}

__device__ int g_gemv_error;   // sticky device error word of this translation unit

// A group whose largest |x| is 2^100 or more (or not finite) is outside the
// staging's exponent range: the call reports it, and its y is undefined.
__device__ __forceinline__ void check_stage_range(float mx) {
    if (!(mx < 0x1p100f)) report_device_error(&g_gemv_error, kDevErrGemvActivationRange);
}

// Scales of a slice [gA, gB): the copy starts at group g_lo and is `width`
// groups wide; 16-byte chunks when every slice starts and ends on a multiple
// of 8 groups, 4-byte pairs when G is even, single halves otherwise.
__host__ __device__ inline int scale_mode(int G, int gA, int gB) {
    if (G % 8 == 0 && gA % 8 == 0 && (gB - gA) % 8 == 0) return 16;
    return G % 2 == 0 ? 4 : 2;
}
__host__ __device__ inline int scale_lo(int G, int gA, int gB) { return scale_mode(G, gA, gB) == 4 ? (gA & ~1) : gA; }
__host__ __device__ inline int scale_width(int G, int gA, int gB) {
    return scale_mode(G, gA, gB) == 4 ? ((gB + 1) & ~1) - (gA & ~1) : gB - gA;
}

// ---- the fused rotation's slice ----
constexpr int kRotN = 1024;                      // a K-slice of 8 groups
constexpr int kRotPitch = kRotN + kRotN / 16;    // floats per token, padded as fwht_pos pads
// This CTA's slice sigma (8 groups) of x' = H_4096 (s (.) x) / 64 for every
// token, into rot[m][fwht_pos(j)], j = 0..1023.  With the block b = sigma / 4
// and the slice's place a = sigma % 4 in it, and H_4096 = H_4 (x) H_1024,
//   x'[4096 b + 1024 a + j] = (H_1024 u)[j],
//   u[j] = sum_{a'} (-1)^popcount(a & a') z[4096 b + 1024 a' + j] / 64,  z = s (.) x.
// H_1024 = H_4 (x) H_16 (x) H_16 runs as three passes (index bits 0-3, 4-7,
// 8-9).  Four tokens at a time, 64 threads each.  All threads of the CTA
// call it; it ends with a barrier.
__device__ __forceinline__ void rotate_slice(const __nv_bfloat16* __restrict__ x, const int8_t* __restrict__ signs,
                                             int K, int M, int sigma, float* __restrict__ rot) {
    const int blk = sigma >> 2, a = sigma & 3;
    const int tq = threadIdx.x >> 6, tau = threadIdx.x & 63;
    for (int m0 = 0; m0 < M; m0 += 4) {
        const int m = m0 + tq;
        float* u = rot + (size_t)m * kRotPitch;
        float v[16];
        if (m < M) {
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] = 0.0f;
#pragma unroll
            for (int ap = 0; ap < 4; ++ap) {
                const size_t k0 = (size_t)kFwhtN * blk + (size_t)kRotN * ap + 16 * tau;
                const int4* xp = reinterpret_cast<const int4*>(x + (size_t)m * K + k0);
                const int4 x0 = __ldg(xp), x1 = __ldg(xp + 1);
                const int4 sg = __ldg(reinterpret_cast<const int4*>(signs + k0));
                const uint32_t xw[8] = {(uint32_t)x0.x, (uint32_t)x0.y, (uint32_t)x0.z, (uint32_t)x0.w,
                                        (uint32_t)x1.x, (uint32_t)x1.y, (uint32_t)x1.z, (uint32_t)x1.w};
                const uint32_t sw[4] = {(uint32_t)sg.x, (uint32_t)sg.y, (uint32_t)sg.z, (uint32_t)sg.w};
                const bool flip = (__popc(a & ap) & 1) != 0;
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const float xv = __uint_as_float(((xw[e >> 1] >> (16 * (e & 1))) & 0xFFFFu) << 16);
                    const int sv = (int)(int8_t)((sw[e >> 2] >> (8 * (e & 3))) & 0xFFu);
                    v[e] += ((sv < 0) != flip) ? -xv : xv;
                }
            }
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] *= 1.0f / 64.0f;
            fwht16(v);   // index bits 0-3
#pragma unroll
            for (int e = 0; e < 16; ++e) u[fwht_pos(16 * tau + e)] = v[e];
        }
        __syncthreads();
        if (m < M) {
            // index bits 4-7: tau's bits 0-3 and 4-5 are bits 0-3 and 8-9
            const int base = (tau & 15) | ((tau >> 4) << 8);
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] = u[fwht_pos(base | (e << 4))];
            fwht16(v);
#pragma unroll
            for (int e = 0; e < 16; ++e) u[fwht_pos(base | (e << 4))] = v[e];
        }
        __syncthreads();
        if (m < M) {
            // index bits 8-9: four columns (bits 0-7) per thread
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
                const int c = 4 * tau + c4;
                const float w0 = u[fwht_pos(c)], w1 = u[fwht_pos(c | 256)];
                const float w2 = u[fwht_pos(c | 512)], w3 = u[fwht_pos(c | 768)];
                const float p0 = w0 + w1, p1 = w0 - w1, p2 = w2 + w3, p3 = w2 - w3;
                u[fwht_pos(c)] = p0 + p2;
                u[fwht_pos(c | 256)] = p1 + p3;
                u[fwht_pos(c | 512)] = p0 - p2;
                u[fwht_pos(c | 768)] = p1 - p3;
            }
        }
        __syncthreads();
    }
}

// ONE: the single-token case (M = 1), whose epilogue keeps one value per row.
// LEAN (when G is a multiple of 8): every warp has exactly one group over its
// CTA's whole range, and only the lean loop is compiled.
// BIN: the 1-bit sibling format (lean loop only): slice sigma is groups
// 8 sigma .. 8 sigma + 7, and a warp whose group is past G has no units.
// AFF: an affine pack, w = s q + b (one matrix, bf16 activations).
template <int MT, bool PRE, bool ONE, bool LEAN = false, bool BIN = false, bool AFF = false, bool ROT = false>
__global__ void __launch_bounds__(kThreads, GemvCfg<MT>::kCtasPerSm)
gemv_kernel(const GemvArgs a) {
    static_assert(!BIN || (LEAN && !PRE), "the 1-bit layout runs the lean loop on bf16 activations");
    static_assert(!ROT || (LEAN && !PRE), "the in-kernel rotation's slices are whole 8-group slices");
    static_assert(!AFF || (!BIN && !PRE), "the affine pack has 2-bit codes and bf16 activations");
    constexpr int MP = 8 * MT;
    constexpr int SLOT = BIN ? kBinSlotBytes : kSlotBytes;
    extern __shared__ __align__(16) unsigned char smem[];
    const int M = ONE ? 1 : a.M;
    const int G = a.G, S = a.S, rmax = a.rmax, gpad = a.gpad;
    const int W = a.K / (BIN ? 32 : 16);   // code words per row
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gid = lane >> 2, t = lane & 3;
    const int sigma = blockIdx.x / a.cps, clu = blockIdx.x - sigma * a.cps;   // slice, range
    // the matrix this range belongs to (a pair call's ranges never straddle the two)
    const bool second = clu >= a.cps1;
    const uint32_t* const codes = second ? a.codes2 : a.codes;
    const __half* const scales = second ? a.scales2 : a.scales;
    float* const yv = second ? a.y2 : a.y;
    const int N = second ? a.N2 : a.N;
    const int Tm = second ? a.T2 : a.T;
    const int cpsm = second ? a.cps - a.cps1 : a.cps1;
    const int clm = second ? clu - a.cps1 : clu;
    const int gA = BIN ? kWarps * sigma : (int)((long long)G * sigma / S);
    const int gB = BIN ? min(gA + kWarps, G) : (int)((long long)G * (sigma + 1) / S);
    const int Gs = gB - gA;
    const int tile_lo = (int)((long long)Tm * clm / cpsm);
    const int R = (int)((long long)Tm * (clm + 1) / cpsm) - tile_lo;
    const int na = Gs / kWarps, nb = Gs - na * kWarps, nseg = na + nb;
    const int g_lo = scale_lo(G, gA, gB);

    unsigned short* sc = reinterpret_cast<unsigned short*>(smem + a.off_sc);   // [R * 16][gpad]
    float* part = reinterpret_cast<float*>(smem + a.off_part);

    // segment s of this warp: s < na is group gA + warp + 8 s over all R tiles;
    // s >= na is left-over group gA + 8 na + (s - na) over tile chunk
    // (warp + s - na) mod 8 (the chunk rotates so no warp takes every short one)
    auto seg_group = [&](int s) { return s < na ? gA + warp + kWarps * s : gA + kWarps * na + (s - na); };
    auto seg_lo = [&](int s) { return s < na ? 0 : R * ((warp + s - na) & 7) / kWarps; };
    auto seg_hi = [&](int s) { return s < na ? R : R * (((warp + s - na) & 7) + 1) / kWarps; };

    // ---- this warp's ring: unit u in slot u mod kDepth; lane l copies row l/2,
    // 16-byte half l%2 of the unit's 32 bytes ----
    unsigned char* ring = smem + (size_t)warp * kDepth * SLOT;
    const uint32_t ring_s = smem_addr(ring) + (uint32_t)lane * 16u;
    const int crow = lane >> 1;
    const size_t cstep = (size_t)16 * W;   // words from one tile to the next
    // issue cursor: segment, units left in it, this lane's next row and source
    int is = 0, ileft = 0, irow = 0;
    const uint32_t* iptr = codes;
    auto iseg_begin = [&](int s) {
        while (s < nseg && seg_lo(s) >= seg_hi(s)) ++s;
        is = s;
        if (s < nseg) {
            const int lo = seg_lo(s);
            ileft = seg_hi(s) - lo;
            irow = (tile_lo + lo) * 16 + crow;
            iptr = codes + (size_t)irow * W + seg_group(s) * 8 + (lane & 1) * 4;
        }
    };
    iseg_begin(0);
    auto issue = [&](int slot) {
        if (is < nseg) {
            const bool ok = irow < N;
            cp_async16(ring_s + (uint32_t)(slot * kSlotBytes), ok ? iptr : codes, ok);
            iptr += cstep;
            irow += 16;
            if (--ileft == 0) iseg_begin(is + 1);
        }
        cp_async_commit();   // one group per unit, empty past the end, so the waits count uniformly
    };

    pdl_launch_dependents();
    // Codes and scales are never the previous kernel's output: the range's
    // scales (one commit group) and the first kEarly units of every warp go
    // out before the PDL wait, the others once the warp has staged its
    // activation (a warp held up issuing copies is late to stage).
    {
        const int row0 = tile_lo * 16, rows = R * 16;
        const int mode = scale_mode(G, gA, gB);
        // the range's [rows][gpad] block of one per-group array (scales, or an
        // affine pack's biases at `dst`)
        auto stage_groups = [&](const __half* src, unsigned short* dst) {
            const uint32_t dst_s = smem_addr(dst);
            if (mode == 16) {
                const int cpr = Gs / 8;
                for (int i = threadIdx.x; i < rows * cpr; i += kThreads) {
                    const int r = i / cpr, c = i - r * cpr;
                    const bool ok = row0 + r < N;
                    cp_async16(dst_s + (uint32_t)(r * gpad + 8 * c) * 2u,
                               ok ? src + (size_t)(row0 + r) * G + gA + 8 * c : src, ok);
                }
            } else if (mode == 4) {
                const int cpr = scale_width(G, gA, gB) / 2;
                for (int i = threadIdx.x; i < rows * cpr; i += kThreads) {
                    const int r = i / cpr, c = i - r * cpr;
                    const bool ok = row0 + r < N;
                    cp_async4(dst_s + (uint32_t)(r * gpad + 2 * c) * 2u,
                              ok ? src + (size_t)(row0 + r) * G + g_lo + 2 * c : src, ok);
                }
            } else {
                for (int i = threadIdx.x; i < rows * Gs; i += kThreads) {
                    const int r = i / Gs, c = i - r * Gs;
                    dst[r * gpad + c] = row0 + r < N ? __half_as_ushort(src[(size_t)(row0 + r) * G + gA + c])
                                                     : (unsigned short)0;
                }
            }
        };
        stage_groups(scales, sc);
        if (AFF) stage_groups(a.biases, sc + a.boff);
        cp_async_commit();
    }
    // the lean loop's refill: unit u of the warp's group is tile u of the range
    // (rows past N read row N - 1; their sums are never written to y).  Lane l
    // copies row l / 2, half l % 2 of the unit's 32 (2-bit) or 16 (1-bit) bytes.
    const int lean_g = gA + warp;
    const bool lean_has = !BIN || lean_g < gB;
    const uint32_t* src_base = codes + (size_t)lean_g * (BIN ? 4 : 8) + (lane & 1) * (BIN ? 2 : 4);
    const int crow0 = tile_lo * 16 + crow;
    const uint32_t ring_lane = smem_addr(ring) + (uint32_t)lane * (BIN ? 8u : 16u);
    auto refill = [&](int u, int slot_) {
        if (lean_has && u < R) {
            const int r = min(crow0 + 16 * u, N - 1);
            if (BIN) cp_async8(ring_lane + (uint32_t)(slot_ * SLOT), src_base + (size_t)r * W);
            else cp_async16(ring_lane + (uint32_t)(slot_ * SLOT), src_base + (size_t)r * W, true);
        }
        cp_async_commit();
    };
#pragma unroll
    for (int i = 0; i < kEarly; ++i) {
        if (BIN) refill(i, i);
        else issue(i);
    }
    pdl_wait();
    // y of the range starts at zero: the slice-0 CTA clears it (after the PDL
    // wait, since the previous kernel may still read y) and counts itself into
    // the range's flag once the zeros are visible to the whole GPU
    // (the lean loop issues the clearing stores here but fences and counts a
    // ring turn later, when the stores have long landed, instead of holding
    // the CTA at a barrier now)
    __shared__ unsigned cleared_warps;
    if (S > 1 && sigma == 0) {
        const int row0 = tile_lo * 16, nrow = min(R * 16, N - row0);
        for (int i = threadIdx.x; i < M * nrow; i += kThreads) {
            const int m = i / nrow, r = i - m * nrow;
            yv[(size_t)m * N + row0 + r] = 0.0f;
        }
        if (!LEAN) {
            __threadfence();
            __syncthreads();
            if (threadIdx.x == 0) red_inc(a.flag + clu, (unsigned)(S - 1));
        } else if (threadIdx.x == 0) {
            cleared_warps = 0u;   // published to the other warps by the barrier below
        }
    }
    // a lean slice-0 warp: its clearing stores are visible; the eighth to say
    // so counts the range's clearing into the flag
    auto count_cleared = [&]() {
        __threadfence();
        __syncwarp();
        if (lane == 0 && atomicAdd(&cleared_warps, 1u) == (unsigned)(kWarps - 1))
            red_inc(a.flag + clu, (unsigned)(S - 1));
    };
    // private partials: a warp's first segment (when it spans the range) stores
    // every tile, later ones add; with no such segment, or with shared atomics,
    // start from zeros
    const int part_n = M <= kPrivateMaxM ? kWarps * rmax * 16 * M : rmax * 16 * MP;
    if (M > kPrivateMaxM || na == 0)
        for (int i = threadIdx.x; i < part_n; i += kThreads) part[i] = 0.0f;
    // the in-kernel rotation: this CTA's slice of x' (after the PDL wait
    // above: x may be the previous kernel's output), built while the first
    // weight copies are still landing
    // (one token: all 256 threads on its slice, five radix-4 passes)
    if (ROT) {
        float* rot = reinterpret_cast<float*>(smem + a.off_rot);
        if (ONE)
            fwht1024_slice(reinterpret_cast<const __nv_bfloat16*>(a.x) + (size_t)(sigma >> 2) * kFwhtN,
                           a.signs + (size_t)(sigma >> 2) * kFwhtN, sigma & 3, rot);
        else
            rotate_slice(reinterpret_cast<const __nv_bfloat16*>(a.x), a.signs, a.K, M, sigma, rot);
    }

    // ---- stage one group's activation (read from global memory, possibly the
    // previous kernel's output): lane (gid, t) holds token nt*8+gid,
    // k = 32t .. 32t+31 of the group, as fp16 x 2^(E + 10 - 2j') with E from
    // the token's largest |x| in the group (the rotation prologue of the fused
    // call has done this already: PRE) ----
    uint32_t b[MT][16];
    float4 f[MT];   // (F, F*acc1) of tokens 2t and 2t+1 of each token tile
    auto stage = [&](int g) {
#pragma unroll
        for (int nt = 0; nt < MT; ++nt) {
            // one staged token: every lane reads token 0 (the other lanes' B
            // columns belong to tokens that do not exist; their results are
            // never read)
            const int m = (ONE && PRE) ? 0 : nt * 8 + gid;
            int E = 0;
            if (PRE) {
                if (m < M) {
                    const uint4* s4 = reinterpret_cast<const uint4*>(
                        reinterpret_cast<const uint32_t*>(a.x) + ((size_t)(m * G + g) * 4 + t) * 16);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint4 u = s4[q];
                        b[nt][4 * q] = u.x;
                        b[nt][4 * q + 1] = u.y;
                        b[nt][4 * q + 2] = u.z;
                        b[nt][4 * q + 3] = u.w;
                    }
                    E = a.xe[m * G + g];
                } else {
#pragma unroll
                    for (int q = 0; q < 16; ++q) b[nt][q] = 0u;
                }
            } else {
                float v[32];
                if (ROT && m < M) {
                    // the rotated slice in shared memory (fp32): one token's
                    // as fwht1024_slice leaves it, several tokens' at kRotPitch
                    const int j0 = (g - gA) * kGroup + 32 * t;
                    if (ONE) {
                        const float4* u4 = reinterpret_cast<const float4*>(
                            reinterpret_cast<const float*>(smem + a.off_rot) + fwht_slice_pos(j0));
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const float4 z = u4[q];
                            v[4 * q] = z.x;
                            v[4 * q + 1] = z.y;
                            v[4 * q + 2] = z.z;
                            v[4 * q + 3] = z.w;
                        }
                    } else {
                        const float* u = reinterpret_cast<const float*>(smem + a.off_rot) + (size_t)m * kRotPitch;
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] = u[fwht_pos(j0 + e)];
                    }
                } else if (m < M) {
                    const uint4* s4 = reinterpret_cast<const uint4*>(
                        reinterpret_cast<const __nv_bfloat16*>(a.x) + (size_t)m * a.K + (size_t)g * kGroup + 32 * t);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint4 u = s4[q];
                        const uint32_t uw[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            v[8 * q + 2 * e] = __uint_as_float(uw[e] << 16);
                            v[8 * q + 2 * e + 1] = __uint_as_float(uw[e] & 0xFFFF0000u);
                        }
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = 0.0f;
                }
                float mx = 0.0f;
#pragma unroll
                for (int e = 0; e < 32; ++e) mx = fmaxf(mx, fabsf(v[e]));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                check_stage_range(mx);
                E = stage_exponent(mx);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    __half2 lo, hi;
                    if (BIN) {
                        // MMA j takes slots j (k = 32t+j, +16) and j + 8 (k = 32t+j+8, +24)
                        const float c0 = bin_stage_multiplier(E, j), c1 = bin_stage_multiplier(E, j + 8);
                        lo = __floats2half2_rn(v[j] * c0, v[j + 16] * c0);
                        hi = __floats2half2_rn(v[j + 8] * c1, v[j + 24] * c1);
                    } else {
                        const float c = stage_multiplier<AFF>(E, j);
                        lo = __floats2half2_rn(v[j] * c, v[j + 8] * c);       // k = 32t+j, +8
                        hi = __floats2half2_rn(v[j + 16] * c, v[j + 24] * c); // k = 32t+16+j, +24
                    }
                    b[nt][2 * j] = *reinterpret_cast<const uint32_t*>(&lo);
                    b[nt][2 * j + 1] = *reinterpret_cast<const uint32_t*>(&hi);
                }
            }
            // the -1 correction: the same chain on the all-ones pattern; every row of
            // the result is the same, lane (gid, t) holds tokens 2t, 2t+1
            // (the 1-bit layout: w = (2b - 1) s, so y = s F (2 acc - acc1))
            float acc1[4];
            if (BIN) {
                bin_chain1(acc1, 0xFFFFFFFFu, 0xFFFFFFFFu, b[nt]);
            } else {
                const uint32_t ones[4] = {0x55555555u, 0x55555555u, 0x55555555u, 0x55555555u};
                mma_chain1<AFF>(acc1, ones, b[nt]);
            }
            const float F = (m < M) ? __uint_as_float((uint32_t)(14 - E + 127) << 23) : 0.0f;   // 2^(14-E)
            const float F0 = __shfl_sync(0xffffffffu, F, (2 * t) * 4);
            const float F1 = __shfl_sync(0xffffffffu, F, (2 * t + 1) * 4);
            constexpr float kq = BIN ? 2.0f : 1.0f;
            f[nt] = make_float4(kq * F0, F0 * acc1[0], kq * F1, F1 * acc1[1]);
        }
    };

    // ---- one unit's rows into the partials: sp = this lane's scale of row gid,
    // pw = the unit's private partial rows (M <= 4) ----
    auto epilogue = [&](auto add_c, const unsigned short* sp, float* pw, int i, const float (&acc)[MT][4]) {
        constexpr bool ADD = decltype(add_c)::value;
        const float s0 = __half2float(__ushort_as_half(sp[0]));
        const float s1 = __half2float(__ushort_as_half(sp[8 * gpad]));
        // one output: s F acc - s F acc1, or s F acc + b F acc1 for an affine pack
        float b0 = 0.0f, b1 = 0.0f;
        if (AFF) {
            b0 = __half2float(__ushort_as_half(sp[a.boff]));
            b1 = __half2float(__ushort_as_half(sp[a.boff + 8 * gpad]));
        }
        auto out = [&](float s_, float b_, float F_, float a_, float Fa1) {
            return AFF ? fmaf(s_ * F_, a_, b_ * Fa1) : s_ * fmaf(F_, a_, -Fa1);
        };
        if (ONE) {
            // token 0 sits in lanes t == 0, element 0 (row gid) and 2 (row gid + 8)
            const float v0 = out(s0, b0, f[0].x, acc[0][0], f[0].y);
            const float v2 = out(s1, b1, f[0].x, acc[0][2], f[0].y);
            if (t == 0) {
                pw[gid] = ADD ? pw[gid] + v0 : v0;
                pw[gid + 8] = ADD ? pw[gid + 8] + v2 : v2;
            }
            return;
        }
#pragma unroll
        for (int nt = 0; nt < MT; ++nt) {
            const int m0 = nt * 8 + 2 * t, m1 = m0 + 1;
            const float v0 = out(s0, b0, f[nt].x, acc[nt][0], f[nt].y);   // row gid,     token m0
            const float v1 = out(s0, b0, f[nt].z, acc[nt][1], f[nt].w);   // row gid,     token m1
            const float v2 = out(s1, b1, f[nt].x, acc[nt][2], f[nt].y);   // row gid + 8, token m0
            const float v3 = out(s1, b1, f[nt].z, acc[nt][3], f[nt].w);   // row gid + 8, token m1
            if (M <= kPrivateMaxM) {
                // [warp][tile][row][M], written only by its warp
                if (m0 < M) {
                    pw[gid * M + m0] = ADD ? pw[gid * M + m0] + v0 : v0;
                    pw[(gid + 8) * M + m0] = ADD ? pw[(gid + 8) * M + m0] + v2 : v2;
                }
                if (m1 < M) {
                    pw[gid * M + m1] = ADD ? pw[gid * M + m1] + v1 : v1;
                    pw[(gid + 8) * M + m1] = ADD ? pw[(gid + 8) * M + m1] + v3 : v3;
                }
            } else {
                float* row = part + (size_t)i * 16 * MP;   // [tile][row][MP], shared by the warps
                if (m0 < M) {
                    atomicAdd(row + gid * MP + m0, v0);
                    atomicAdd(row + (gid + 8) * MP + m0, v2);
                }
                if (m1 < M) {
                    atomicAdd(row + gid * MP + m1, v1);
                    atomicAdd(row + (gid + 8) * MP + m1, v3);
                }
            }
        }
    };

    // ---- the segments ----
    int slot = 0;   // ring slot of the next unit to consume
    const unsigned char* rd = ring + gid * (BIN ? 16 : 32) + (BIN ? 4 : 8) * t;   // this lane's words in a slot
    const int sstep = 16 * gpad;                          // scale halves per tile
    const int pstep = 16 * M;                             // private partial floats per tile
    auto run_segment = [&](auto add_c, int lo, int hi, int g) {
        const unsigned short* sp = sc + (lo * 16 + gid) * gpad + (g - g_lo);
        float* pw = part + ((size_t)warp * rmax + lo) * pstep;
        for (int i = lo; i < hi; i += 2) {
            const bool two = i + 1 < hi;
            const int slot1 = slot + 1 == kDepth ? 0 : slot + 1;
            // units i and i + 1 have landed (at most kDepth - 2 newer groups pending)
            cp_async_wait<kDepth - 2>();
            __syncwarp();
            uint32_t w[2][4];
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const unsigned char* sp8 = rd + (q ? slot1 : slot) * kSlotBytes;
                const uint2 v0 = *reinterpret_cast<const uint2*>(sp8);
                const uint2 v1 = *reinterpret_cast<const uint2*>(sp8 + 8 * 32);
                w[q][0] = v0.x;   // row gid,     word 2t      (MMA rows 0-7,  k-slots 2t, 2t+1)
                w[q][1] = v1.x;   // row gid + 8, word 2t      (MMA rows 8-15)
                w[q][2] = v0.y;   // row gid,     word 2t + 1  (k-slots 2t+8, 2t+9)
                w[q][3] = v1.y;   // row gid + 8, word 2t + 1
            }
            float acc[2][MT][4];
            if (two) {
                pair_mmas<MT, AFF>(acc, w, b);
            } else {
#pragma unroll
                for (int nt = 0; nt < MT; ++nt) mma_chain1<AFF>(acc[0][nt], w[0], b[nt]);
            }
            // the consumed slots are fully read by every lane: refill them kDepth units ahead
            __syncwarp();
            issue(slot);
            if (two) issue(slot1);
            epilogue(add_c, sp, pw, i, acc[0]);
            if (two) epilogue(add_c, sp + sstep, pw + pstep, i + 1, acc[1]);
            sp += 2 * sstep;
            pw += 2 * pstep;
            slot = two ? (slot1 + 1 == kDepth ? 0 : slot1 + 1) : slot1;
        }
    };
    // this thread's scale copies (the oldest group) have landed; after the
    // barrier every thread's have, and the zeroed partials are visible
    static_assert(kEarly >= 2 && kEarly <= kDepth && kDepth % 2 == 0, "ring accounting");
    cp_async_wait<kEarly>();
    __syncthreads();
    // the range's flag, read ahead so the load overlaps the loop (a slice other
    // than 0 needs it non-zero before adding into y); the lean loop reads it a
    // ring turn in, after the slice-0 CTA has had time to clear y
    const bool flag_reader = S > 1 && sigma != 0 && threadIdx.x == 0;
    unsigned flag_seen = 0u;
    if (!LEAN && flag_reader) flag_seen = ld_acquire_gpu(a.flag + clu);
    if (LEAN) {
        // The common case: one group per warp over the whole range (K a
        // multiple of 1024, or any K for the 1-bit layout).  Whole turns of the
        // ring run with compile-time slots, and a refill's source is the row
        // base plus a per-tile stride.
        const int g = lean_g;
        const bool clearer = S > 1 && sigma == 0;
        if (!lean_has) {
            // a warp with no group (the last slice of a 1-bit K that is not a
            // multiple of 1024): its partials stay zero
            if (clearer) count_cleared();
        } else {
        stage(g);
#pragma unroll
        for (int u = kEarly; u < kDepth; ++u) {
            if (BIN) refill(u, u);
            else issue(u);
        }
        const unsigned short* sp = sc + gid * gpad + (g - g_lo);
        float* pw = part + (size_t)warp * rmax * pstep;   // private partials (M <= 4)
        auto fast_step = [&](int i, int s0, int s1, bool two) {
            cp_async_wait<kDepth - 2>();
            __syncwarp();
            float acc[2][MT][4];
            if constexpr (BIN) {
                uint32_t w[2][2];
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const unsigned char* sp8 = rd + (q ? s1 : s0) * SLOT;
                    w[q][0] = *reinterpret_cast<const uint32_t*>(sp8);            // row gid,     word t
                    w[q][1] = *reinterpret_cast<const uint32_t*>(sp8 + 8 * 16);   // row gid + 8, word t
                }
                if (two) {
                    bin_pair_mmas<MT>(acc, w, b);
                } else {
#pragma unroll
                    for (int nt = 0; nt < MT; ++nt) bin_chain1(acc[0][nt], w[0][0], w[0][1], b[nt]);
                }
            } else {
                uint32_t w[2][4];
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const unsigned char* sp8 = rd + (q ? s1 : s0) * SLOT;
                    const uint2 v0 = *reinterpret_cast<const uint2*>(sp8);
                    const uint2 v1 = *reinterpret_cast<const uint2*>(sp8 + 8 * 32);
                    w[q][0] = v0.x;
                    w[q][1] = v1.x;
                    w[q][2] = v0.y;
                    w[q][3] = v1.y;
                }
                if (two) {
                    pair_mmas<MT, AFF>(acc, w, b);
                } else {
#pragma unroll
                    for (int nt = 0; nt < MT; ++nt) mma_chain1<AFF>(acc[0][nt], w[0], b[nt]);
                }
            }
            __syncwarp();
            refill(i + kDepth, s0);
            if (two) refill(i + 1 + kDepth, s1);
            epilogue(std::false_type{}, sp, pw, i, acc[0]);
            if (two) epilogue(std::false_type{}, sp + sstep, pw + pstep, i + 1, acc[1]);
            sp += 2 * sstep;
            pw += 2 * pstep;
        };
        bool counted = false;
        int i = 0;
        for (; i + kDepth <= R; i += kDepth) {
            if (i == kDepth) {
                if (flag_reader) flag_seen = ld_acquire_gpu(a.flag + clu);
                if (clearer) {
                    count_cleared();
                    counted = true;
                }
            }
#pragma unroll
            for (int q = 0; q < kDepth; q += 2) fast_step(i + q, q, q + 1, true);
        }
        for (int q = 0; i < R; i += 2, q += 2) fast_step(i, q, q + 1, i + 1 < R);
        if (clearer && !counted) count_cleared();   // a range of less than two ring turns
        }
    } else {
        bool rest_issued = false;
        for (int s = 0; s < nseg; ++s) {
            const int lo = seg_lo(s), hi = seg_hi(s);
            if (lo >= hi) continue;
            const int g = seg_group(s);
            stage(g);
            if (!rest_issued) {
#pragma unroll
                for (int u = kEarly; u < kDepth; ++u) issue(u);
                rest_issued = true;
            }
            if (s > 0 && na > 0) run_segment(std::true_type{}, lo, hi, g);
            else run_segment(std::false_type{}, lo, hi, g);
        }
    }
    cp_async_wait<0>();
    __syncthreads();

    // ---- the CTA's row sums ----
    const int nr = R * 16;
    auto row_value = [&](int tl, int r, int m) -> float {
        if (M <= kPrivateMaxM) {
            float s = 0.0f;
            for (int w2 = 0; w2 < kWarps; ++w2) s += part[(((size_t)w2 * rmax + tl) * 16 + r) * M + m];
            return s;
        }
        return part[((size_t)tl * 16 + r) * MP + m];
    };
    if (S == 1) {
        for (int m = 0; m < M; ++m)
            for (int rr = threadIdx.x; rr < nr; rr += kThreads) {
                const int r = tile_lo * 16 + rr;
                if (r < N) yv[(size_t)m * N + r] = row_value(rr >> 4, rr & 15, m);
            }
        return;
    }
    // ---- several slices: add the CTA's row sums into y.  A slice other than 0
    // first waits (bounded) until the slice-0 CTA has cleared the rows -- it
    // cleared them right after the PDL wait and counted a ring turn later at
    // most, so by now the count has normally been seen -- and counts itself;
    // the S-th count returns the flag to 0. ----
    __shared__ int go;
    if (sigma != 0) {
        if (threadIdx.x == 0) {
            const bool ok = flag_seen != 0u || wait_flag_nonzero(a.flag + clu, kFlagWaitNs);
            if (ok) red_inc(a.flag + clu, (unsigned)(S - 1));
            else report_device_error(&g_gemv_error, kDevErrGemvConsumerWait);
            go = ok;
        }
        __syncthreads();
        if (!go) return;   // reported: y is left incomplete rather than wrong-ordered
    }
    for (int m = 0; m < M; ++m)
        for (int rr = threadIdx.x; rr < nr; rr += kThreads) {
            const int r = tile_lo * 16 + rr;
            if (r < N) atomicAdd(yv + (size_t)m * N + r, row_value(rr >> 4, rr & 15, m));
        }
}

// Rotation prologue for the fused path: x' = H_4096 (s (.) x) / 64 in fp32,
// staged for the product exactly as the product stages a bf16 x (per token and
// group, E from the largest |x'| and fp16 x' 2^(E + 10 - 2j')), so x' is never
// rounded to bf16.  One CTA per (token, 1024-wide slice sigma of a 4096-block
// b = sigma / 4), with H_4096 = H_4 (x) H_1024 in natural order: the slice is
// H_1024 u, u[j] = sum_{a'} (-1)^popcount(a & a') z[4096 b + 1024 a' + j] / 64
// (a = sigma % 4, z = s (.) x).  The fragments are stored in
// the order the product's lanes hold them: xs[m][g][t][r] (uint32, two
// halves), lane t's B register r; xe[m][g] = E.  Threads 0-63 stage: thread i
// owns the slice's values 16 i .. 16 i + 15, one half of lane t's registers of
// one group.
__global__ void __launch_bounds__(kFwhtThreads)
rotate_stage_kernel(const __nv_bfloat16* __restrict__ x, const int8_t* __restrict__ signs,
                    uint32_t* __restrict__ xs, int* __restrict__ xe, int K) {
    __shared__ __align__(16) float sm[kFwhtSliceSmemFloats];
    pdl_launch_dependents();
    pdl_wait();
    const int sigma = blockIdx.x, m = blockIdx.y, G = K / kGroup;
    const int blk = sigma >> 2;
    const int i = threadIdx.x;
    fwht1024_slice(x + (size_t)m * K + (size_t)blk * kFwhtN, signs + (size_t)blk * kFwhtN, sigma & 3, sm);
    if (i >= 64) return;
    float v[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) v[e] = sm[fwht_slice_pos(16 * i + e)];
    float mx = 0.0f;
#pragma unroll
    for (int e = 0; e < 16; ++e) mx = fmaxf(mx, fabsf(v[e]));
    // the eight threads of a group are lanes 8c .. 8c + 7 of one warp
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
    check_stage_range(mx);
    const int E = stage_exponent(mx);
    const int g = sigma * (kRotN / kGroup) + (i >> 3);
    const int e0 = 16 * (i & 7);                    // first value within the group
    const int t = e0 >> 5, half = (e0 >> 4) & 1;    // lane t; this thread forms its registers 2j + half
    uint32_t r[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float c = stage_multiplier(E, j);
        const __half2 h = __floats2half2_rn(v[j] * c, v[j + 8] * c);
        r[j] = *reinterpret_cast<const uint32_t*>(&h);
    }
    // the thread pair of lane t swaps halves so that each stores eight
    // consecutive registers: half 0 registers 0-7, half 1 registers 8-15
    uint32_t o[8];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint32_t got = __shfl_xor_sync(0xffffffffu, half ? r[q] : r[q + 4], 1);
        o[2 * q] = half ? got : r[q];
        o[2 * q + 1] = half ? r[q + 4] : got;
    }
    uint4* dst = reinterpret_cast<uint4*>(xs + ((size_t)(m * G + g) * 4 + t) * 16 + 8 * half);
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
    if ((i & 7) == 0) xe[m * G + g] = E;
}

// ---------------------------------------------------------------------------
// The product for 5 to 16 tokens, tile-major (2-bit codes, K a multiple of 256).
//
// Above, with several tokens every (tile, group) unit writes M partial row
// sums per row to shared memory (with shared atomics past four tokens) and
// eight warps' partials are summed at the end; that bookkeeping grows with M
// while the MMAs do not.  Here a warp owns whole 16-row tiles and walks the
// CTA's K-slice over them, two tiles and two groups (one 2 KB stage of codes
// and the tiles' 32 x 2 scales) at a time, keeping the tiles' 16 x M sums in
// registers, so each output is written once; each group's staged activation
// is read once for both tiles.  The slice's staged activation
// is computed once per CTA into shared memory, in the lanes' B-fragment order
// (the same fp16 x 2^(E + 10 - 2j') values as above), with the all-ones
// correction of each (group, token tile) and the tokens' F beside it.  The
// MMA of a unit and of the ones pass compute each output from the same A row
// and B column in the same order, so a row of zero weights gives exactly 0.
// ---------------------------------------------------------------------------
constexpr int kTDuo = 2;                                       // groups per stage
constexpr int kTDepth = 4;                                     // stages in flight per warp (a power of 2)
constexpr int kTCodeBytes = 2 * kTDuo * kSlotBytes;            // one stage's codes: [group][tile] 16 x 32-byte units
constexpr int kTStageBytes = kTCodeBytes + 32 * kTDuo * 2;     // and the two tiles' 32 x 2 scales
constexpr int kTRingBytes = kWarps * kTDepth * kTStageBytes;
constexpr int kTFragBytes = 4 * 32 * 16;                       // one (group, token tile): [4][32 lanes][16 B]
constexpr int kTCorrBytes = 4 * 16;                            // (F, F acc1) of tokens 2t, 2t + 1: [4 t][float4]
constexpr int kTCtasPerSm = 2;
// staging items per warp whose loads go out together (one token tile; with
// two, the extra registers spill)
template <int MT> struct TStage { static constexpr int kBatch = MT == 1 ? 3 : 1; };
// From five tokens on (where the product above turns to shared atomics) the
// tile-major loop is the faster one; from two, also for matrices of at most
// kTileSmallN rows (measured on 5120 -> 6144: 6.54 / 6.56 us at two / four
// tokens against 6.80 / 7.37; on 5120 -> 17408 the product above stays ahead).
constexpr int kTileMinM = 5;
constexpr int kTileSmallN = 8192;

// A unit's chains for all MT token tiles, each slot unpacked once for all.
template <int MT>
__device__ __forceinline__ void unit_chains(float (&acc)[MT][4], const uint32_t (&w)[4], const uint32_t (&b)[MT][16]) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        uint32_t r[4];
        slot_regs<false>(j, w[0], w[1], w[2], w[3], r);
#pragma unroll
        for (int nt = 0; nt < MT; ++nt)
            mma16816(acc[nt], r[0], r[1], r[2], r[3], b[nt][2 * j], b[nt][2 * j + 1], j > 0);
    }
}

template <int MT, bool PRE>
__global__ void __launch_bounds__(kThreads, kTCtasPerSm) gemvt_kernel(const GemvArgs a) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int M = a.M, G = a.G, S = a.S;
    const int W = a.K / 16;   // code words per row
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gid = lane >> 2, t = lane & 3;
    const int sigma = blockIdx.x / a.cps, clu = blockIdx.x - sigma * a.cps;   // slice, range
    const bool second = clu >= a.cps1;
    const uint32_t* const codes = second ? a.codes2 : a.codes;
    const __half* const scales = second ? a.scales2 : a.scales;
    float* const yv = second ? a.y2 : a.y;
    const int N = second ? a.N2 : a.N;
    const int Tm = second ? a.T2 : a.T;
    const int cpsm = second ? a.cps - a.cps1 : a.cps1;
    const int clm = second ? clu - a.cps1 : clu;
    // slice sigma: duos [qA, qA + nq) of the row's G / 2 group pairs
    const int Gq = G / kTDuo;
    const int qA = (int)((long long)Gq * sigma / S);
    const int nq = (int)((long long)Gq * (sigma + 1) / S) - qA;
    const int gA = kTDuo * qA, Gs = kTDuo * nq;
    // the range's tile pairs (tiles 2p and 2p + 1; a second tile past the
    // matrix has rows past N); warp w takes pairs w, w + 8, ... of it
    const int Pm = (Tm + 1) >> 1;
    const int pair_lo = (int)((long long)Pm * clm / cpsm);
    const int R = (int)((long long)Pm * (clm + 1) / cpsm) - pair_lo;
    const int n_items = warp < R ? (R - 1 - warp) / kWarps + 1 : 0;
    const int n_st = n_items * nq;

    unsigned char* const ring = smem + (size_t)warp * kTDepth * kTStageBytes;
    unsigned char* const frag = smem + kTRingBytes;                                  // [Gs][MT][4][32][16 B]
    unsigned char* const corr = frag + (size_t)Gs * MT * kTFragBytes;                // [Gs][MT][4][float4]

    // ---- this warp's copies: stage s is duo s % nq of item s / nq.  Lane l
    // copies 16-byte half l % 2 of row l / 2 of each (group, tile) unit, and
    // the 4 bytes of scales of the pair's row l.  Rows past N read row N - 1;
    // their sums are never written. ----
    const uint32_t ring_s = smem_addr(ring);
    const uint32_t dst_c = (uint32_t)((lane >> 1) * 32 + (lane & 1) * 16);
    const uint32_t dst_s = (uint32_t)(kTCodeBytes + lane * 4);
    const uint32_t* src_c[2];
    const __half* src_s = scales;
    int i_item = 0, i_q = 0, issued = 0;
    auto item_src = [&](int it) {
        const int row0 = (pair_lo + warp + kWarps * it) * 32;
#pragma unroll
        for (int tau = 0; tau < 2; ++tau)
            src_c[tau] = codes + (size_t)min(row0 + 16 * tau + (lane >> 1), N - 1) * W + (size_t)gA * 8 + (lane & 1) * 4;
        src_s = scales + (size_t)min(row0 + lane, N - 1) * G + gA;
    };
    src_c[0] = src_c[1] = codes;
    if (n_items > 0) item_src(0);
    auto issue = [&](int slot) {
        if (issued < n_st) {
            const uint32_t base = ring_s + (uint32_t)(slot * kTStageBytes);
#pragma unroll
            for (int g = 0; g < kTDuo; ++g)
#pragma unroll
                for (int tau = 0; tau < 2; ++tau)
                    cp_async16(base + (uint32_t)((2 * g + tau) * kSlotBytes) + dst_c, src_c[tau] + 8 * g, true);
            src_c[0] += kTDuo * 8;
            src_c[1] += kTDuo * 8;
            cp_async4(base + dst_s, src_s, true);
            src_s += kTDuo;
            ++issued;
            if (++i_q == nq) {
                i_q = 0;
                if (++i_item < n_items) item_src(i_item);
            }
        }
        cp_async_commit();   // one group per stage, empty past the end, so the waits count uniformly
    };

    pdl_launch_dependents();
    // codes and scales are never the previous kernel's output: the first
    // stages go out before the PDL wait
#pragma unroll
    for (int i = 0; i < kTDepth; ++i) issue(i);
    pdl_wait();

    // ---- several slices: the slice-0 CTA clears the range's rows of y (each
    // warp the rows of its own tiles) and counts itself into the range's flag
    // once every warp's zeros are visible; a CTA of another slice adds only
    // after its warps have seen the flag non-zero, and counts itself once all
    // of them have; the S-th count returns the flag to 0. ----
    __shared__ unsigned cleared_warps, seen_warps;
    const bool clearer = S > 1 && sigma == 0;
    const bool adder = S > 1 && sigma != 0;
    if (threadIdx.x == 0) {
        cleared_warps = 0u;
        seen_warps = 0u;
    }
    if (clearer)
        for (int it = 0; it < n_items; ++it) {
            const int r = (pair_lo + warp + kWarps * it) * 32 + lane;
            if (r < N)
                for (int m = 0; m < M; ++m) yv[(size_t)m * N + r] = 0.0f;
        }

    // ---- stage the slice's activation: item (g, nt) of the Gs x MT, warp w
    // taking items w, w + 8, ...; lane (gid, t) holds token 8 nt + gid,
    // values 32 t .. 32 t + 31 of group gA + g, exactly as the product above
    // stages a group ----
    {
        // a warp's items go kBatch at a time, their loads issued
        // together so that one round trip serves them all
        const __nv_bfloat16* x = reinterpret_cast<const __nv_bfloat16*>(a.x);
        const int n_items_x = Gs * MT;
        for (int base = warp; base < n_items_x; base += kWarps * TStage<MT>::kBatch) {
        uint4 raw[TStage<MT>::kBatch][4];
        int raw_e[TStage<MT>::kBatch];
#pragma unroll
        for (int j = 0; j < TStage<MT>::kBatch; ++j) {
            const int item = base + j * kWarps;
            const int g = item / MT, nt = item - g * MT;
            const int m = nt * 8 + gid;
            raw_e[j] = 0;
            if (PRE && item < n_items_x && m < M) raw_e[j] = a.xe[m * G + gA + g];
            if (item < n_items_x && m < M) {
                const uint4* s4 =
                    PRE ? reinterpret_cast<const uint4*>(reinterpret_cast<const uint32_t*>(a.x) +
                                                         ((size_t)(m * G + gA + g) * 4 + t) * 16)
                        : reinterpret_cast<const uint4*>(x + (size_t)m * a.K + (size_t)(gA + g) * kGroup + 32 * t);
#pragma unroll
                for (int q = 0; q < 4; ++q) raw[j][q] = s4[q];
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q) raw[j][q] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
#pragma unroll
        for (int j = 0; j < TStage<MT>::kBatch; ++j) {
            const int item = base + j * kWarps;
            if (item >= n_items_x) break;
            int E = 0;
            uint32_t b[16];
            if (PRE) {
                // the fragments and exponent as the rotation prologue staged them
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    b[4 * q] = raw[j][q].x;
                    b[4 * q + 1] = raw[j][q].y;
                    b[4 * q + 2] = raw[j][q].z;
                    b[4 * q + 3] = raw[j][q].w;
                }
                E = raw_e[j];
            } else {
            float v[32];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint32_t uw[4] = {raw[j][q].x, raw[j][q].y, raw[j][q].z, raw[j][q].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    v[8 * q + 2 * e] = __uint_as_float(uw[e] << 16);
                    v[8 * q + 2 * e + 1] = __uint_as_float(uw[e] & 0xFFFF0000u);
                }
            }
            float mx = 0.0f;
#pragma unroll
            for (int e = 0; e < 32; ++e) mx = fmaxf(mx, fabsf(v[e]));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            check_stage_range(mx);
            E = stage_exponent(mx);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float c = stage_multiplier(E, j);
                const __half2 lo = __floats2half2_rn(v[j] * c, v[j + 8] * c);        // k = 32t+j, +8
                const __half2 hi = __floats2half2_rn(v[j + 16] * c, v[j + 24] * c);  // k = 32t+16+j, +24
                b[2 * j] = *reinterpret_cast<const uint32_t*>(&lo);
                b[2 * j + 1] = *reinterpret_cast<const uint32_t*>(&hi);
            }
            }
            unsigned char* fp = frag + (size_t)item * kTFragBytes + lane * 16;
#pragma unroll
            for (int q = 0; q < 4; ++q)
                *reinterpret_cast<uint4*>(fp + q * 512) = make_uint4(b[4 * q], b[4 * q + 1], b[4 * q + 2], b[4 * q + 3]);
            // the all-ones pass: column n is token 8 nt + n; lane (., t) holds
            // tokens 2t and 2t + 1, whose F the lanes of rows 2t and 2t + 1 hold
            float acc1[4];
            const uint32_t ones[4] = {0x55555555u, 0x55555555u, 0x55555555u, 0x55555555u};
            unit_chain(acc1, ones, b);
            const float F = __uint_as_float((uint32_t)(14 - E + 127) << 23);   // 2^(14-E)
            const float F0 = __shfl_sync(0xffffffffu, F, (2 * t) * 4);
            const float F1 = __shfl_sync(0xffffffffu, F, (2 * t + 1) * 4);
            if (gid == 0)
                *reinterpret_cast<float4*>(corr + ((size_t)item * 4 + t) * 16) =
                    make_float4(F0, F0 * acc1[0], F1, F1 * acc1[1]);
        }
        }
    }
    __syncthreads();

    // a slice-0 warp: its clearing stores are visible; the eighth to say so
    // counts the range's clearing into the flag
    auto count_cleared = [&]() {
        __threadfence();
        __syncwarp();
        if (lane == 0 && atomicAdd(&cleared_warps, 1u) == (unsigned)(kWarps - 1))
            red_inc(a.flag + clu, (unsigned)(S - 1));
    };
    auto count_seen = [&]() {
        if (lane == 0 && atomicAdd(&seen_warps, 1u) == (unsigned)(kWarps - 1))
            red_inc(a.flag + clu, (unsigned)(S - 1));
    };
    if (clearer && n_st == 0) count_cleared();
    if (adder && n_st == 0) count_seen();   // a warp with tiles counts once it has seen the flag

    // ---- the stages ----
    const unsigned char* const rd = ring + gid * 32 + 8 * t;   // this lane's words of row gid in a stage's unit 0
    unsigned flag_seen = 0u;
    bool add_ok = true;
    int s = 0;
    for (int it = 0; it < n_items; ++it) {
        // rows gid and gid + 8 of tiles 2p and 2p + 1, tokens 8 nt + 2t and 8 nt + 2t + 1
        float y[2][MT][4];
#pragma unroll
        for (int tau = 0; tau < 2; ++tau)
#pragma unroll
            for (int nt = 0; nt < MT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) y[tau][nt][e] = 0.0f;
        for (int q = 0; q < nq; ++q, ++s) {
            const int slot = s & (kTDepth - 1);
            // stage s has landed (at most kTDepth - 1 newer groups pending)
            cp_async_wait<kTDepth - 1>();
            __syncwarp();
            const unsigned char* st = rd + slot * kTStageBytes;
            const unsigned char* scp = ring + slot * kTStageBytes + kTCodeBytes;
            // the scales of rows gid and gid + 8 of both tiles, both groups
            float sv[2][2][kTDuo];
#pragma unroll
            for (int tau = 0; tau < 2; ++tau)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float2 f2 =
                        __half22float2(*reinterpret_cast<const __half2*>(scp + (16 * tau + 8 * h + gid) * 4));
                    sv[tau][h][0] = f2.x;
                    sv[tau][h][1] = f2.y;
                }
#pragma unroll
            for (int g = 0; g < kTDuo; ++g) {
                const int gl = kTDuo * q + g;
                // the group's staged activation, read once for both tiles
                uint32_t b[MT][16];
                float4 f[MT];
#pragma unroll
                for (int nt = 0; nt < MT; ++nt) {
                    const unsigned char* fp = frag + (size_t)(gl * MT + nt) * kTFragBytes + lane * 16;
#pragma unroll
                    for (int qq = 0; qq < 4; ++qq) {
                        const uint4 z = *reinterpret_cast<const uint4*>(fp + qq * 512);
                        b[nt][4 * qq] = z.x;
                        b[nt][4 * qq + 1] = z.y;
                        b[nt][4 * qq + 2] = z.z;
                        b[nt][4 * qq + 3] = z.w;
                    }
                    f[nt] = *reinterpret_cast<const float4*>(corr + ((size_t)(gl * MT + nt) * 4 + t) * 16);
                }
#pragma unroll
                for (int tau = 0; tau < 2; ++tau) {
                    const unsigned char* up = st + (2 * g + tau) * kSlotBytes;
                    const uint2 v0 = *reinterpret_cast<const uint2*>(up);
                    const uint2 v1 = *reinterpret_cast<const uint2*>(up + 8 * 32);
                    // row gid word 2t, row gid + 8 word 2t, then words 2t + 1
                    const uint32_t w[4] = {v0.x, v1.x, v0.y, v1.y};
                    float acc[MT][4];
                    unit_chains<MT>(acc, w, b);
                    const float sa = sv[tau][0][g], sb = sv[tau][1][g];
#pragma unroll
                    for (int nt = 0; nt < MT; ++nt) {
                        y[tau][nt][0] = fmaf(sa, fmaf(f[nt].x, acc[nt][0], -f[nt].y), y[tau][nt][0]);   // row gid,     token 2t
                        y[tau][nt][1] = fmaf(sa, fmaf(f[nt].z, acc[nt][1], -f[nt].w), y[tau][nt][1]);   // row gid,     token 2t+1
                        y[tau][nt][2] = fmaf(sb, fmaf(f[nt].x, acc[nt][2], -f[nt].y), y[tau][nt][2]);   // row gid + 8, token 2t
                        y[tau][nt][3] = fmaf(sb, fmaf(f[nt].z, acc[nt][3], -f[nt].w), y[tau][nt][3]);   // row gid + 8, token 2t+1
                    }
                }
            }
            // the stage is fully read by every lane: refill it kTDepth stages ahead
            __syncwarp();
            issue(slot);
            if (s == 0) {
                if (clearer) count_cleared();
                // read ahead, so the load overlaps the loop
                if (adder && lane == 0) flag_seen = ld_acquire_gpu(a.flag + clu);
            }
        }
        // the tiles' sums
        if (adder && it == 0) {
            int ok = 1;
            if (lane == 0) {
                ok = flag_seen != 0u || wait_flag_nonzero(a.flag + clu, kFlagWaitNs);
                if (!ok) report_device_error(&g_gemv_error, kDevErrGemvConsumerWait);
            }
            add_ok = __shfl_sync(0xffffffffu, ok, 0) != 0;
            if (add_ok) count_seen();
        }
        if (add_ok) {
            const int row0 = (pair_lo + warp + kWarps * it) * 32 + gid;
#pragma unroll
            for (int tau = 0; tau < 2; ++tau)
#pragma unroll
                for (int nt = 0; nt < MT; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int m = nt * 8 + 2 * t + (e & 1), r = row0 + 16 * tau + 8 * (e >> 1);
                        if (m < M && r < N) {
                            float* p = yv + (size_t)m * N + r;
                            if (S == 1) *p = y[tau][nt][e];
                            else atomicAdd(p, y[tau][nt][e]);
                        }
                    }
        }
    }
    cp_async_wait<0>();
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
struct Plan {
    int G, T, S, cps, ctas, rmax, MT, gpad, slot;
    int T2, cps1;   // a pair call: the second matrix's tiles (T counts both) and the first's ranges
    bool aff;       // an affine pack: biases staged after the scales, boff halves on
    bool rot;       // the in-kernel rotation (ROT): the rotated slice after the partials
    int boff;
    uint32_t off_sc, off_part, off_rot;
    size_t smem;
};

// Shared-memory layout for `cps` ranges (ring | scales | biases (AFF) | partials).
// `cps` ranges over T tiles (the last T2 of them a pair call's second matrix):
// returns the longest range, sets the first matrix's range count.  A pair
// call's ranges are shared out in proportion to the tiles, at least one each,
// so no range straddles the two matrices.
int split_ranges(int T, int T2, int& cps, int& cps1) {
    if (T2 > 0) {
        const int T1 = T - T2;
        cps = std::max(cps, 2);
        cps1 = std::min(cps - 1, std::max(1, (int)(((long long)cps * T1 + T / 2) / T)));
        return std::max((T1 + cps1 - 1) / cps1, (T2 + cps - cps1 - 1) / (cps - cps1));
    }
    cps1 = cps;
    return (T + cps - 1) / cps;
}

void layout(Plan& p, int M, int cps) {
    p.rmax = split_ranges(p.T, p.T2, cps, p.cps1);
    p.cps = cps;
    const int MP = 8 * p.MT;
    size_t off = (size_t)kWarps * kDepth * p.slot;
    p.off_sc = (uint32_t)off;
    p.boff = p.rmax * 16 * p.gpad;   // a multiple of 8 halves: 16-byte aligned
    off = align_up(off + (size_t)p.rmax * 16 * p.gpad * 2 * (p.aff ? 2 : 1), 16);
    p.off_part = (uint32_t)off;
    off += (M <= kPrivateMaxM ? (size_t)kWarps * p.rmax * 16 * M : (size_t)p.rmax * 16 * MP) * 4;
    p.off_rot = (uint32_t)align_up(off, 16);
    if (p.rot) off = p.off_rot + (M == 1 ? (size_t)kFwhtSliceSmemFloats : (size_t)M * kRotPitch) * 4;
    p.smem = off;
}

// The device-independent part of the plan: slices and the scale pitch.  The
// 1-bit layout's slices are groups 8 s .. 8 s + 7 (the last one may be short).
Plan base_plan(int M, int N, int K, bool bin, int N2 = 0, bool aff = false, bool rot = false) {
    Plan p{};
    p.aff = aff;
    p.rot = rot;
    p.G = K / kGroup;
    p.T2 = (N2 + 15) / 16;
    p.T = (N + 15) / 16 + p.T2;
    p.S = (p.G + kWarps - 1) / kWarps;
    p.MT = (M + 7) / 8;
    p.slot = bin ? kBinSlotBytes : kSlotBytes;
    int w = 0;
    for (int s = 0; s < p.S; ++s) {
        const int gA = bin ? kWarps * s : (int)((long long)p.G * s / p.S);
        const int gB = bin ? std::min(gA + kWarps, p.G) : (int)((long long)p.G * (s + 1) / p.S);
        w = std::max(w, scale_width(p.G, gA, gB));
    }
    p.gpad = (int)align_up((size_t)w, 8);   // row pitch a multiple of 16 bytes
    return p;
}

// Lets the kernel use the device's whole per-block shared memory; returns the
// dynamic part it may take.
template <int MT, bool PRE, bool ONE, bool LEAN, bool BIN, bool AFF, bool ROT>
cudaError_t kernel_smem_limit(int dev, int* limit) {
    static int optin_of[64] = {};
    if (!optin_of[dev]) {
        int optin = 0;
        cudaError_t e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e != cudaSuccess) return e;
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, gemv_kernel<MT, PRE, ONE, LEAN, BIN, AFF, ROT>);
        if (e != cudaSuccess) return e;
        optin -= (int)fa.sharedSizeBytes;   // the kernel's static shared memory comes first
        e = cudaFuncSetAttribute(gemv_kernel<MT, PRE, ONE, LEAN, BIN, AFF, ROT>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
        if (e != cudaSuccess) return e;
        optin_of[dev] = optin;
    }
    *limit = optin_of[dev];
    return cudaSuccess;
}

// One wave: as many CTAs as fit at once, by registers (the launch bound) and
// by shared memory (which grows with the range length).
template <int MT, bool PRE, bool ONE, bool LEAN, bool BIN, bool AFF, bool ROT>
tern_status make_plan(int M, int N, int K, int N2, int sms, int dev, Plan* out) {
    int limit = 0;
    if (kernel_smem_limit<MT, PRE, ONE, LEAN, BIN, AFF, ROT>(dev, &limit) != cudaSuccess) return TERN_ERR_CUDA;
    Plan p = base_plan(M, N, K, BIN, N2, AFF, ROT);
    const int need = (p.T + kMaxTiles - 1) / kMaxTiles;   // ranges short enough for the shared partials
    int cps = 1;
    for (int per_sm = GemvCfg<MT>::kCtasPerSm; per_sm >= 1; --per_sm) {
        cps = std::max(need, std::min(p.T, std::max(1, sms * per_sm / p.S)));
        layout(p, M, cps);
        if ((size_t)per_sm * (p.smem + kCtaSmemReserve) <= kSmemPerSm) break;
    }
    // very long slices: shorter ranges (more than one wave) until a CTA fits
    while (p.smem > (size_t)limit && p.rmax > 1)
        layout(p, M, std::max(p.cps + 1, (p.T + p.rmax - 2) / (p.rmax - 1) + (p.T2 > 0 ? 1 : 0)));
    if (p.smem > (size_t)limit) return TERN_ERR_SHAPE;
    p.ctas = p.S * p.cps;
    *out = p;
    return TERN_OK;
}

// Plans depend on the shape and the device only: keep the recent ones.
struct PlanKey {
    int M, N, K, N2, dev;
    bool pre, bin, aff, rot;
};
std::mutex g_plan_mu;
constexpr int kPlanCache = 64;
PlanKey g_plan_key[kPlanCache];
Plan g_plan_val[kPlanCache];
int g_plan_n = 0, g_plan_next = 0;

template <int MT, bool PRE, bool ONE, bool LEAN, bool BIN, bool AFF, bool ROT>
tern_status cached_plan(int M, int N, int K, int N2, int sms, Plan* out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TERN_ERR_CUDA;
    if (dev < 0 || dev >= 64) return TERN_ERR_DEVICE;
    std::lock_guard<std::mutex> lk(g_plan_mu);
    for (int i = 0; i < g_plan_n; ++i) {
        const PlanKey& k = g_plan_key[i];
        if (k.M == M && k.N == N && k.K == K && k.N2 == N2 && k.dev == dev && k.pre == PRE && k.bin == BIN &&
            k.aff == AFF && k.rot == ROT) {
            *out = g_plan_val[i];
            return TERN_OK;
        }
    }
    const tern_status st = make_plan<MT, PRE, ONE, LEAN, BIN, AFF, ROT>(M, N, K, N2, sms, dev, out);
    if (st != TERN_OK) return st;
    const int slot = g_plan_n < kPlanCache ? g_plan_n++ : (g_plan_next++ % kPlanCache);
    g_plan_key[slot] = PlanKey{M, N, K, N2, dev, PRE, BIN, AFF, ROT};
    g_plan_val[slot] = *out;
    return TERN_OK;
}

// ---- the tile-major product for 2 to 16 tokens: slices of whole quads,
// ranges of tiles, one wave of CTAs when it fits ----
struct PlanT {
    int S, cps, cps1, ctas;
    size_t smem;
};
size_t smem_t(int Gs, int MT) { return (size_t)kTRingBytes + (size_t)Gs * MT * (kTFragBytes + kTCorrBytes); }

// The slice count trades the longest warp's stages (a warp's tiles times the
// slice's quads) against the extra CTAs and the additions into y that more
// slices bring, within the shared memory the slice's staged activation
// needs; the range flags exist only when K spans more than one 1024-wide
// slice, so shorter K keeps one slice.
template <int MT, bool PRE>
tern_status make_plan_t(int N, int K, int N2, int sms, int dev, PlanT* out) {
    static int optin_of[64] = {};
    if (!optin_of[dev]) {
        int optin = 0;
        if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
            return TERN_ERR_CUDA;
        cudaFuncAttributes fa;
        if (cudaFuncGetAttributes(&fa, gemvt_kernel<MT, PRE>) != cudaSuccess) return TERN_ERR_CUDA;
        optin -= (int)fa.sharedSizeBytes;
        if (cudaFuncSetAttribute(gemvt_kernel<MT, PRE>, cudaFuncAttributeMaxDynamicSharedMemorySize, optin) !=
            cudaSuccess)
            return TERN_ERR_CUDA;
        optin_of[dev] = optin;
    }
    // ranges over tile pairs, slices over group pairs
    const int G = K / kGroup, Gq = G / kTDuo;
    const int T2 = ((N2 + 15) / 16 + 1) / 2, T = ((N + 15) / 16 + 1) / 2 + T2;
    double best = 0.0;
    PlanT bp{};
    for (int S = 1; S <= Gq && S <= 64; ++S) {
        if (S > 1 && G <= kWarps) break;
        const int qmax = (Gq + S - 1) / S;
        const size_t sm = smem_t(kTDuo * qmax, MT);
        if (sm > (size_t)optin_of[dev]) continue;
        const int per_sm = std::min(kTCtasPerSm, (int)(kSmemPerSm / (sm + kCtaSmemReserve)));
        if (per_sm < 1) continue;
        const int slots = sms * per_sm;
        int cps = std::max(1, std::min(T, slots / S)), cps1 = 0;
        const int rmax = split_ranges(T, T2, cps, cps1);
        const int items = (rmax + kWarps - 1) / kWarps;
        const long long waves = ((long long)S * cps + slots - 1) / slots;
        const double cost = (double)waves * (items * (qmax + 1.0) + 2.0 + (S > 1 ? 1.0 : 0.0));
        if (bp.ctas == 0 || cost < best) {
            best = cost;
            bp = PlanT{S, cps, cps1, S * cps, sm};
        }
    }
    if (bp.ctas == 0) return TERN_ERR_SHAPE;
    *out = bp;
    return TERN_OK;
}

struct PlanTKey {
    int MT, N, K, N2, dev;
    bool pre;
};
PlanTKey g_plant_key[kPlanCache];
PlanT g_plant_val[kPlanCache];
int g_plant_n = 0, g_plant_next = 0;

template <int MT, bool PRE>
tern_status cached_plan_t(int N, int K, int N2, int sms, PlanT* out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TERN_ERR_CUDA;
    if (dev < 0 || dev >= 64) return TERN_ERR_DEVICE;
    std::lock_guard<std::mutex> lk(g_plan_mu);
    for (int i = 0; i < g_plant_n; ++i) {
        const PlanTKey& k = g_plant_key[i];
        if (k.MT == MT && k.N == N && k.K == K && k.N2 == N2 && k.dev == dev && k.pre == PRE) {
            *out = g_plant_val[i];
            return TERN_OK;
        }
    }
    const tern_status st = make_plan_t<MT, PRE>(N, K, N2, sms, dev, out);
    if (st != TERN_OK) return st;
    const int slot = g_plant_n < kPlanCache ? g_plant_n++ : (g_plant_next++ % kPlanCache);
    g_plant_key[slot] = PlanTKey{MT, N, K, N2, dev, PRE};
    g_plant_val[slot] = *out;
    return TERN_OK;
}

template <int MT, bool PRE = false>
tern_status launch_gemv_t(GemvArgs args, int sms, cudaStream_t stream) {
    PlanT p;
    const tern_status st = cached_plan_t<MT, PRE>(args.N, args.K, args.N2, sms, &p);
    if (st != TERN_OK) return st;
    args.G = args.K / kGroup;
    args.T = (args.N + 15) / 16;
    args.T2 = (args.N2 + 15) / 16;
    args.S = p.S;
    args.cps = p.cps;
    args.cps1 = p.cps1;
    const cudaError_t e =
        launch_pdl(gemvt_kernel<MT, PRE>, dim3(p.ctas), dim3(kThreads), p.smem, stream, true, args);
    return e == cudaSuccess ? TERN_OK : TERN_ERR_CUDA;
}

tern_status validate(const void* x, const uint32_t* codes, const void* scales, const float* y, int M, int N, int K) {
    if (M < 1 || M > 16 || N < 1 || K < kGroup || K % kGroup != 0) return TERN_ERR_SHAPE;
    if ((long long)N * (K / 16) >= (1LL << 40) || (long long)M * K >= (1LL << 31) || N >= (1 << 28))
        return TERN_ERR_SHAPE;
    if (!x || !codes || !scales || !y) return TERN_ERR_NULL;
    if (!aligned16(x) || !aligned16(codes) || !aligned16(scales) || !aligned16(y)) return TERN_ERR_ALIGN;
    return TERN_OK;
}

// Workspace: [range flag words, when K spans several slices | the staged
// rotated x, for the rotation-fused call].  The flags count back to 0 at the end of every
// call, so a zero-filled workspace stays ready for the next one.
size_t flag_bytes(int N, int K) {
    const int G = K / kGroup;
    return G > kWarps ? align_up((size_t)((N + 15) / 16) * 4, 256) : 0;
}
// The range flags of a call over T 16-row tiles (one matrix, or both of a
// pair call), when K spans several slices.
size_t base_bytes(int M, int T, int K) {
    (void)M;
    const int G = K / kGroup;
    return G > kWarps ? align_up((size_t)T * 4, 256) : 0;
}
// The in-kernel rotation (ROT) serves M <= kRotMaxM; above that the fused call
// stages the rotated x in the workspace.
constexpr int kRotMaxM = 2;
size_t workspace_bytes(int M, int N, int K, bool rot) {
    if (M < 1 || M > 16 || N < 1 || K < kGroup || K % kGroup != 0) return 0;
    return base_bytes(M, (N + 15) / 16, K) +
           (rot && M > kRotMaxM ? align_up((size_t)M * K * 2 + (size_t)M * (K / kGroup) * 4, 256) : 0);
}

template <int MT, bool PRE, bool ONE, bool LEAN = false, bool BIN = false, bool AFF = false, bool ROT = false>
tern_status launch_gemv(GemvArgs args, int sms, cudaStream_t stream) {
    Plan p;
    const tern_status st = cached_plan<MT, PRE, ONE, LEAN, BIN, AFF, ROT>(args.M, args.N, args.K, args.N2, sms, &p);
    if (st != TERN_OK) return st;
    args.G = p.G;
    args.T = p.T - p.T2;   // the first matrix's tiles
    args.T2 = p.T2;
    args.cps1 = p.cps1;
    args.S = p.S;
    args.cps = p.cps;
    args.rmax = p.rmax;
    args.gpad = p.gpad;
    args.boff = p.boff;
    args.off_sc = p.off_sc;
    args.off_part = p.off_part;
    args.off_rot = p.off_rot;
    const cudaError_t e =
        launch_pdl(gemv_kernel<MT, PRE, ONE, LEAN, BIN, AFF, ROT>, dim3(p.ctas), dim3(kThreads), p.smem, stream, true,
                   args);
    return e == cudaSuccess ? TERN_OK : TERN_ERR_CUDA;
}

tern_status run(const void* x, const int8_t* signs, const uint32_t* codes, const void* scales, float* y, int M,
                int N, int K, void* workspace, size_t workspace_bytes_, cudaStream_t stream, bool bin = false,
                const uint32_t* codes2 = nullptr, const void* scales2 = nullptr, float* y2 = nullptr, int N2 = 0,
                const void* biases = nullptr) {
    int sms = 0;
    tern_status st = check_device(&sms);
    if (st != TERN_OK) return st;
    const size_t fb = base_bytes(M, (N + 15) / 16 + (N2 + 15) / 16, K);
    if (fb > 0 || signs) {
        const size_t need = fb + (signs ? workspace_bytes(M, N, K, true) - base_bytes(M, (N + 15) / 16, K) : 0);
        if (need > 0 && (!workspace || workspace_bytes_ < need)) return TERN_ERR_WORKSPACE;
        if (reinterpret_cast<uintptr_t>(workspace) & 255u) return TERN_ERR_ALIGN;
    }
    GemvArgs args{};
    args.flag = fb > 0 ? reinterpret_cast<unsigned*>(workspace) : nullptr;
    args.x = x;
    args.codes = codes;
    args.scales = reinterpret_cast<const __half*>(scales);
    args.biases = reinterpret_cast<const __half*>(biases);
    args.y = y;
    args.M = M;
    args.N = N;
    args.K = K;
    args.codes2 = N2 > 0 ? codes2 : codes;
    args.scales2 = reinterpret_cast<const __half*>(N2 > 0 ? scales2 : scales);
    args.y2 = N2 > 0 ? y2 : y;
    args.N2 = N2;
    const int MT = (M + 7) / 8;
    // K a multiple of 1024: slices of exactly 8 groups, one group per warp
    const bool lean = (K / kGroup) % kWarps == 0;
    int launches = 1;
    if (signs && M <= kRotMaxM) {
        // the rotation inside the product (K % 4096 == 0: whole 8-group slices)
        args.signs = signs;
        st = M == 1 ? launch_gemv<1, false, true, true, false, false, true>(args, sms, stream)
                    : launch_gemv<1, false, false, true, false, false, true>(args, sms, stream);
    } else if (signs) {
        // staged x': M x K halves, then M x G exponents
        uint32_t* xs = reinterpret_cast<uint32_t*>(reinterpret_cast<char*>(workspace) + fb);
        int* xe = reinterpret_cast<int*>(xs + (size_t)M * K / 2);
        const cudaError_t e = launch_pdl(rotate_stage_kernel, dim3(K / kRotN, M), dim3(kFwhtThreads), 0, stream,
                                         true, reinterpret_cast<const __nv_bfloat16*>(x), signs, xs, xe, K);
        if (e != cudaSuccess) return TERN_ERR_CUDA;
        args.x = xs;
        args.xe = xe;
        launches = 2;
        if (M >= kTileMinM || N <= kTileSmallN)
            st = MT == 1 ? launch_gemv_t<1, true>(args, sms, stream) : launch_gemv_t<2, true>(args, sms, stream);
        else
            st = MT == 1 ? launch_gemv<1, true, false, true>(args, sms, stream)
                         : launch_gemv<2, true, false, true>(args, sms, stream);
    } else if (biases) {
        st = M == 1 ? (lean ? launch_gemv<1, false, true, true, false, true>(args, sms, stream)
                            : launch_gemv<1, false, true, false, false, true>(args, sms, stream))
             : MT == 1 ? (lean ? launch_gemv<1, false, false, true, false, true>(args, sms, stream)
                               : launch_gemv<1, false, false, false, false, true>(args, sms, stream))
                       : (lean ? launch_gemv<2, false, false, true, false, true>(args, sms, stream)
                               : launch_gemv<2, false, false, false, false, true>(args, sms, stream));
    } else if (bin) {
        // the 1-bit layout always runs the lean loop
        st = M == 1 ? launch_gemv<1, false, true, true, true>(args, sms, stream)
             : MT == 1 ? launch_gemv<1, false, false, true, true>(args, sms, stream)
                       : launch_gemv<2, false, false, true, true>(args, sms, stream);
    } else if ((M >= kTileMinM || (M >= 2 && N + N2 <= kTileSmallN)) && K % (kTDuo * kGroup) == 0) {
        st = MT == 1 ? launch_gemv_t<1>(args, sms, stream) : launch_gemv_t<2>(args, sms, stream);
    } else {
        st = M == 1 ? (lean ? launch_gemv<1, false, true, true>(args, sms, stream)
                            : launch_gemv<1, false, true>(args, sms, stream))
             : MT == 1 ? (lean ? launch_gemv<1, false, false, true>(args, sms, stream)
                               : launch_gemv<1, false, false>(args, sms, stream))
                       : (lean ? launch_gemv<2, false, false, true>(args, sms, stream)
                               : launch_gemv<2, false, false>(args, sms, stream));
    }
    if (st != TERN_OK) return st;
    set_launch_count(launches);
    return TERN_OK;
}

}  // namespace

// Reads and clears the decode product's device error word (set when a slice's
// bounded wait for its range's clearing gave up).
cudaError_t read_gemv_device_error(int* code) {
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_gemv_error, sizeof(int));
    if (e != cudaSuccess) return e;
    if (v != 0) {
        const int z = 0;
        e = cudaMemcpyToSymbol(g_gemv_error, &z, sizeof(int));
        if (e != cudaSuccess) return e;
    }
    *code = v;
    return cudaSuccess;
}

// The range-flag wait run on a word that nothing ever sets: it gives up after
// limit_ns and reports the code a K-slice reports when the slice-0 CTA never
// counts its clearing of y.
__device__ unsigned g_never_set;   // zero-initialised; no kernel writes it
__global__ void flag_wait_selftest_kernel(uint64_t limit_ns) {
    if (threadIdx.x == 0 && !wait_flag_nonzero(&g_never_set, limit_ns))
        report_device_error(&g_gemv_error, kDevErrGemvConsumerWait);
}
cudaError_t launch_flag_wait_selftest(uint64_t limit_ns, cudaStream_t stream) {
    flag_wait_selftest_kernel<<<1, 32, 0, stream>>>(limit_ns);
    return cudaGetLastError();
}

}  // namespace tern

using namespace tern;

extern "C" size_t tern_gemv_workspace_bytes(int M, int N, int K) {
    // covers both the plain and the rotation-fused call of the same shape
    const size_t b = workspace_bytes(M, N, K, (K % kFwhtN) == 0);
    return b > 0 ? b : (M >= 1 && M <= 16 && N >= 1 && K >= kGroup && K % kGroup == 0 ? 256 : 0);
}

extern "C" tern_status tern_gemv(const void* x, const uint32_t* codes, const void* scales, float* y, int M,
                                 int N, int K, void* workspace, size_t workspace_bytes_, tern_stream_t stream) {
    set_launch_count(0);
    const tern_status v = validate(x, codes, scales, y, M, N, K);
    if (v != TERN_OK) return v;
    const size_t need = workspace_bytes(M, N, K, false);
    if (need > 0 && (!workspace || workspace_bytes_ < need)) return TERN_ERR_WORKSPACE;
    return run(x, nullptr, codes, scales, y, M, N, K, workspace, workspace_bytes_, (cudaStream_t)stream);
}

extern "C" size_t tern_gemv_pair_workspace_bytes(int M, int N_a, int N_b, int K) {
    if (M < 1 || M > 16 || N_a < 1 || N_b < 1 || K < kGroup || K % kGroup != 0) return 0;
    return std::max<size_t>(256, base_bytes(M, (N_a + 15) / 16 + (N_b + 15) / 16, K));
}

extern "C" tern_status tern_gemv_pair(const void* x, const uint32_t* codes_a, const void* scales_a, float* y_a,
                                      int N_a, const uint32_t* codes_b, const void* scales_b, float* y_b, int N_b,
                                      int M, int K, void* workspace, size_t workspace_bytes_, tern_stream_t stream) {
    set_launch_count(0);
    tern_status v = validate(x, codes_a, scales_a, y_a, M, N_a, K);
    if (v != TERN_OK) return v;
    v = validate(x, codes_b, scales_b, y_b, M, N_b, K);
    if (v != TERN_OK) return v;
    if ((long long)N_a + N_b >= (1 << 28)) return TERN_ERR_SHAPE;
    const size_t need = base_bytes(M, (N_a + 15) / 16 + (N_b + 15) / 16, K);
    if (need > 0 && (!workspace || workspace_bytes_ < need)) return TERN_ERR_WORKSPACE;
    return run(x, nullptr, codes_a, scales_a, y_a, M, N_a, K, workspace, workspace_bytes_, (cudaStream_t)stream,
               false, codes_b, scales_b, y_b, N_b);
}

extern "C" tern_status tern_affine_gemv(const void* x, const uint32_t* codes, const void* scales, const void* biases,
                                        float* y, int M, int N, int K, void* workspace, size_t workspace_bytes_,
                                        tern_stream_t stream) {
    set_launch_count(0);
    const tern_status v = validate(x, codes, scales, y, M, N, K);
    if (v != TERN_OK) return v;
    if (!biases) return TERN_ERR_NULL;
    if (!aligned16(biases)) return TERN_ERR_ALIGN;
    const size_t need = workspace_bytes(M, N, K, false);
    if (need > 0 && (!workspace || workspace_bytes_ < need)) return TERN_ERR_WORKSPACE;
    return run(x, nullptr, codes, scales, y, M, N, K, workspace, workspace_bytes_, (cudaStream_t)stream, false,
               nullptr, nullptr, nullptr, 0, biases);
}

extern "C" tern_status tern_bin_gemv(const void* x, const uint32_t* words, const void* scales, float* y, int M,
                                     int N, int K, void* workspace, size_t workspace_bytes_,
                                     tern_stream_t stream) {
    set_launch_count(0);
    const tern_status v = validate(x, words, scales, y, M, N, K);
    if (v != TERN_OK) return v;
    const size_t need = workspace_bytes(M, N, K, false);
    if (need > 0 && (!workspace || workspace_bytes_ < need)) return TERN_ERR_WORKSPACE;
    return run(x, nullptr, words, scales, y, M, N, K, workspace, workspace_bytes_, (cudaStream_t)stream, true);
}

extern "C" tern_status tern_fwht_gemm(const void* x, const int8_t* signs, const uint32_t* codes,
                                      const void* scales, float* y, int M, int N, int K, void* workspace,
                                      size_t workspace_bytes_, tern_stream_t stream) {
    set_launch_count(0);
    if (K % kFwhtN != 0) return TERN_ERR_SHAPE;
    const tern_status v = validate(x, codes, scales, y, M, N, K);
    if (v != TERN_OK) return v;
    if (!signs) return TERN_ERR_NULL;
    if (!aligned16(signs)) return TERN_ERR_ALIGN;
    if (!workspace || workspace_bytes_ < workspace_bytes(M, N, K, true)) return TERN_ERR_WORKSPACE;
    return run(x, signs, codes, scales, y, M, N, K, workspace, workspace_bytes_, (cudaStream_t)stream);
}

// ---------------------------------------------------------------------------
// Decode product with no allocation anywhere.
//
// Some callers cannot allocate device memory for a workspace: code that runs
// where an allocation may not happen (inside a custom allocator's own callback,
// a caching allocator that must not recurse, an embedded runtime that owns all
// device memory up front).  For them the product's only scratch -- the range
// flag words -- lives in one fixed array in the library's own device memory,
// which every GPU that loads the library holds until the process exits.
// ---------------------------------------------------------------------------
namespace tern {
namespace {

constexpr size_t kNoAllocScratchBytes = TERN_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// The device address of the array on the current device.  In host code the
// array's name is only a stand-in for the symbol, so the address comes from
// cudaGetSymbolAddress, with the device current.  It is looked up on every
// call (a host-side query that issues no stream work), so an address can never
// outlive a device reset that reloads the module.
cudaError_t noalloc_scratch(void** out) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    *out = p;
    return cudaSuccess;
}

}  // namespace
}  // namespace tern

extern "C" tern_status tern_gemv_noalloc(const void* x, const uint32_t* codes, const void* scales, float* y, int M,
                                         int N, int K, tern_stream_t stream) {
    set_launch_count(0);
    const tern_status v = validate(x, codes, scales, y, M, N, K);
    if (v != TERN_OK) return v;
    const size_t need = tern::flag_bytes(N, K);
    if (need > kNoAllocScratchBytes) return TERN_ERR_WORKSPACE;
    int sms = 0;
    tern_status st = check_device(&sms);
    if (st != TERN_OK) return st;
    void* scratch = nullptr;
    if (noalloc_scratch(&scratch) != cudaSuccess) return TERN_ERR_CUDA;
    // the flags count back to 0 at the end of every call; clearing them first
    // keeps a call correct even after an earlier one stopped on a device error
    if (need > 0 && cudaMemsetAsync(scratch, 0, need, (cudaStream_t)stream) != cudaSuccess) return TERN_ERR_CUDA;
    return run(x, nullptr, codes, scales, y, M, N, K, scratch, kNoAllocScratchBytes, (cudaStream_t)stream);
}
