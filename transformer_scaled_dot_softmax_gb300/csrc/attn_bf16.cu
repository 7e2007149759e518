// attn_bf16.cu -- fused scaled dot-product attention forward for sm_103a.
//
// Computes, per (batch b, head h), O = softmax(scale * Q K^T + mask) V
// ("Attention Is All You Need" (azimuth.plus), "The idea: every word queries
// every word"; aiany.app Step 6, matrix form S = QK^T/sqrt(d_k),
// A = softmax(S), Z = AV) without ever writing S or A to global memory: the
// softmax is taken online over 128-key tiles (running reference maximum m and
// row sum l, the partial output rescaled when m moves), which reaches the same
// result up to rounding order.
//
// Work item = one 128-row query tile of one (b, h).  The kernel is persistent:
// one CTA per SM walks a static list of items (longest first, dealt to the
// CTAs in snake order so every CTA gets the same number of key tiles), and
// every role runs ahead into the next item as soon as its resources free up,
// so loads, score products and the output of consecutive items overlap.
// Warp roles (16 warps):
//
//   warp 8      TMA producer: Q of each item into one of two Q buffers; K_j and
//               V_j together into a 5-stage ring (one barrier per stage).
//   warp 9      issues S_j = Q K_j^T (tcgen05.mma kind::f16, M=128 N=128,
//               fp32 accumulator in tensor memory).
//   warps 10,11 issue the P.V products of softmax groups A and B into
//               their accumulators O_A and O_B (M = 128, N = 64; A operand P
//               read straight from tensor memory).
//   warps 0-3   softmax group A, warps 4-7 group B: one thread per query row
//               (= tensor-memory lane).  The kernel is a template over how
//               the groups split a row's keys: by key halves (group h takes
//               keys [64h, 64h+64) of every tile; chosen for short items) or
//               by alternate tiles (group A the CTA's even tiles g, group B
//               the odd ones, each tile's 128 scores in two rounds of 64;
//               chosen for long items).
//               Each thread applies the causal / key-padding mask in-tile
//               (masked score = -inf, i.e. exactly zero weight: aiany.app
//               Step 10; notebook chapter "Masked Attention in the Decoder"),
//               keeps its group's reference maximum m_h and sum l_h, and
//               writes P = bf16(2^(s*c - m_h*c)) back over the scores.
//   warps 12-15 output: once an item's products are complete, combine the
//               two groups, normalise, store, and hand the accumulators back.
//
// Splitting a row's keys between two groups with their own maxima, sums and
// accumulators is exact: the output is
//   out = (O_A 2^((m_A-M)c) + O_B 2^((m_B-M)c)) / (l_A 2^((m_A-M)c) + l_B 2^((m_B-M)c)),
// M = max(m_A, m_B).  The groups never wait for each other inside the loop.
// By alternate tiles, the two softmax warps that share a sub-partition work
// one score tile apart instead of in lockstep, so one's tensor-memory round
// trips overlap the other's exponentials; by halves, a one-tile item is
// finished by both groups at once.
//
// MMA issue: one thread can issue a tcgen05.mma only every ~50-80 cycles
// when it runs alone inside `if (lane == 0)`, while an N = 64 product needs
// ~32 cycles of tensor-core time; issued by an elected lane of a converged
// warp with descriptors formed as base + constant, the rate matches the
// tensor core.  Three issuing warps keep S and the two groups' P.V products
// independent of each other.
//
// Score tiles rotate through three tensor-memory buffers (global tile g of
// the CTA in buffer g mod 3): while the softmax works on S_g, S_{g+1} is
// ready and S_{g+2} is being computed.  Issuers are ordered only through
// barriers:
//   S ready (per buffer)           S issuer -> softmax,
//   P ready                        softmax -> PV issuer: by halves per
//                                  (buffer, half); by tiles per (group,
//                                  round), two deep over the group's own
//                                  tiles.  The issuer starts a tile's first
//                                  four products on round 0's P, while the
//                                  softmax works on round 1, and the last
//                                  four on round 1's.  A barrier shared by
//                                  both groups would let one group's issuer
//                                  mistake the other group's unfinished
//                                  phase (parity one behind) for its own
//                                  finished one,
//   round 0 product done (by tiles, per group, two deep)  PV issuer h ->
//                                  softmax group h when round 1 must rescale
//                                  O_h,
//   stage released                 the tile's PV issuer -> TMA producer, S
//                                  issuer (S_g overwrites tile g-3's buffer,
//                                  so it waits for tile g-3's release) and a
//                                  softmax that must rescale O_h (its group's
//                                  previous tile, g-2),
//   Q released (per Q buffer)      S issuer -> TMA producer,
//   output final (count 2)         both PV issuers -> output warps,
//   row statistics (count 8)      softmax -> output warps, and back,
//   accumulators free (count 4)    output warps -> PV issuers.
// A buffer's next use needs its current use to be consumed, so no barrier
// can run two phases ahead of its waiter.
//
// No maximum pass per tile: each round of 64 scores (by halves: a group's
// 64 scores of a tile) is exponentiated against
// the group's current reference maximum (softmax is shift-invariant, so any
// reference that keeps the exponentials finite gives the same result), and
// only a row whose round sum exceeds 2^16 -- its maximum grew by 10 to 16
// log2 units or more -- takes the exact step (round maximum, O_h and l_h
// rescaled -- in round 1 after the round-0 product, taken against the old
// reference, has landed in O_h -- P recomputed).  Unless the log-sum-exp
// is exported, a row's first round is taken against the reference 0 and
// kept if its sum lies in [2^-64, 2^16] (0 then becomes the reference);
// otherwise, or with no visible key, or with lse exported, it takes the
// exact step.  Decided per row.
//
// Tensor memory (512 columns): S buffers [0,128), [128,256), [256,384);
// O_A [384,448), O_B [448,512).  P (bf16, two keys per column) goes over
// scores already read: by tiles into buffer columns [0,64) (round 0 writes
// [0,32), round 1 [32,64)); by halves, half h's 32 columns at [64h, 64h+32).
#include <cuda_bf16.h>

#include <algorithm>

#include "kernels.h"
#include "sm103_ptx.cuh"

namespace mha {
namespace {

constexpr int BM = kAttnRowsPerCta;  // query rows per item
constexpr int BN = 128;              // keys per tile
constexpr int HD = kAttnHeadDim;
constexpr int STAGES = 5;            // K/V ring depth
constexpr int kSBufs = 3;            // score buffers in tensor memory
constexpr int kThreads = 512;        // 8 softmax + load + 3 MMA + 4 output warps
constexpr int kSoftmaxWarps = 8;
constexpr int kLoadWarp = 8;
constexpr int kMmaSWarp = 9;         // issues S = Q K^T
constexpr int kMmaPvWarp = 10;       // warps 10, 11 issue PV for the even / odd tiles
constexpr int kOutWarp = 12;         // warps 12-15: output
constexpr uint32_t kTileBytes = BM * HD * 2;  // 16 KiB, one 128 x 64 bf16 tile
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kOCol = 384;  // O_A [384,448), O_B [448,512)
constexpr float kTileSumLimit = 65536.0f;  // 2^16: a tile sum above it takes the exact step
// A row's first round is tried against the reference 0; a sum below 2^-64
// (the scores far below 0, or none visible) takes the exact step instead.
constexpr float kFirstSumMin = 5.421010862427522e-20f;  // 2^-64
// Per-batch key lengths are read from the CTA's shared-memory copy when it
// holds them all (B <= kLensCache), else from global memory.
constexpr int kLensCache = 1024;
// The geometry of a CTA's first kItemTable items is computed once, in the
// prologue, into shared memory (every role looks each item up).
constexpr int kItemTable = 64;

struct __align__(1024) SmemAttn {
    uint8_t q[2][kTileBytes];
    uint8_t k[STAGES][kTileBytes];
    uint8_t v[STAGES][kTileBytes];
    float red_m[2][BM];  // [group][row]: reference maximum at the end of an item
    float red_l[2][BM];  // [group][row]: row sum at the end of an item
    uint64_t q_full[2];
    uint64_t q_empty[2];
    uint64_t kv_full[STAGES];
    uint64_t kv_empty[STAGES];
    uint64_t s_full[kSBufs];
    uint64_t p_full[kSBufs][2];  // P written (4 warps), by halves: [buffer][half]
    uint64_t p_rd[2][2][2];      // by tiles: [group][round][group tile mod 2], P round written
    uint64_t pv0[2][2];          // by tiles: [group][group tile mod 2], round-0 product complete
    uint64_t ml_full;            // row statistics written (8 softmax warps)
    uint64_t ml_free;            // row statistics read (4 output warps)
    uint64_t o_final;            // both groups' P.V products of an item complete
    uint64_t o_free;             // accumulators read (4 output warps)
    uint64_t drain[3];           // one per MMA-issuing warp
    int lens[kLensCache];        // key_lens[0 .. B) when B <= kLensCache
    int item_tab[kItemTable][6]; // this CTA's first items: bh, b, hh, q0, kv_len, n_kv
    int n_items;                 // items this CTA walks
    uint32_t tmem_base;
    int abort_flag;
};

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }
__device__ __forceinline__ uint32_t f2u(float x) { return __float_as_uint(x); }

// Geometry of one work item.  Items are numbered longest first (query block
// qb from the last down, then (b, h)); round t of the walk gives CTA c the
// item t*G + c (t even) or t*G + G-1-c (t odd).
struct Item {
    int bh, b, hh, q0;
    int kv_len;  // keys [0, kv_len) exist for this batch (padding)
    int n_kv;    // key tiles to visit
};

__device__ __forceinline__ int item_index(int t, int c, int G) {
    return t * G + ((t & 1) ? (G - 1 - c) : c);
}

__device__ __forceinline__ Item make_item(const AttnParams &p, int k, const int *lens_smem) {
    Item it;
    const int BH = p.B * p.H;
    const int qb = p.num_qblocks - 1 - k / BH;
    it.bh = k - (k / BH) * BH;
    it.b = it.bh / p.H;
    it.hh = it.bh - it.b * p.H;
    it.q0 = qb * BM;
    int kv_len = p.Tk;
    if ((p.mask & kMaskPaddingBit) && p.key_lens)
        kv_len = min(max(p.B <= kLensCache ? lens_smem[it.b] : p.key_lens[it.b], 0), p.Tk);
    it.kv_len = kv_len;
    const int kv_end = (p.mask & kMaskCausalBit) ? min(kv_len, min(it.q0 + BM, p.Tq)) : kv_len;
    it.n_kv = (kv_end + BN - 1) / BN;
    return it;
}

__device__ __forceinline__ Item item_of(const SmemAttn &sm, const AttnParams &p, int t, int cta, int G) {
    if (t >= kItemTable) return make_item(p, item_index(t, cta, G), sm.lens);
    Item it;
    it.bh = sm.item_tab[t][0];
    it.b = sm.item_tab[t][1];
    it.hh = sm.item_tab[t][2];
    it.q0 = sm.item_tab[t][3];
    it.kv_len = sm.item_tab[t][4];
    it.n_kv = sm.item_tab[t][5];
    return it;
}

template <bool kTiles, bool kLse>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_bf16_kernel(const __grid_constant__ CUtensorMap tmap_q,
                         const __grid_constant__ CUtensorMap tmap_k,
                         const __grid_constant__ CUtensorMap tmap_v, const AttnParams p) {
    extern __shared__ uint8_t smem_raw[];
    SmemAttn &sm = *reinterpret_cast<SmemAttn *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = static_cast<int>(gridDim.x);
    const int cta = static_cast<int>(blockIdx.x);
    const int total = p.total_items;
    const bool causal = (p.mask & kMaskCausalBit) != 0;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.q_full[i], 1);
            mbar_init(&sm.q_empty[i], 1);
        }
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&sm.kv_full[i], 1);
            mbar_init(&sm.kv_empty[i], kTiles ? 1 : 2);  // the tile's PV issuer(s)
        }
        for (int i = 0; i < kSBufs; ++i) {
            mbar_init(&sm.s_full[i], 1);
            mbar_init(&sm.p_full[i][0], kSoftmaxWarps / 2);
            mbar_init(&sm.p_full[i][1], kSoftmaxWarps / 2);
        }
        for (int i = 0; i < 8; ++i) mbar_init(&sm.p_rd[i >> 2][(i >> 1) & 1][i & 1], kSoftmaxWarps / 2);
        for (int i = 0; i < 4; ++i) mbar_init(&sm.pv0[i >> 1][i & 1], 1);
        mbar_init(&sm.ml_full, kSoftmaxWarps);
        mbar_init(&sm.ml_free, 4);
        mbar_init(&sm.o_final, 2);  // one commit per PV issuer
        mbar_init(&sm.o_free, 4);
        for (int i = 0; i < 3; ++i) mbar_init(&sm.drain[i], 1);
        sm.abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == kMmaSWarp) {
        tmem_alloc(&sm.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    // The key lengths are an input of the call that no kernel of the call
    // writes, so they may be read before waiting for the previous kernel;
    // every role looks them up per item, and a global load there would sit on
    // each item's critical path.
    if ((p.mask & kMaskPaddingBit) && p.key_lens && p.B <= kLensCache)
        for (int i = threadIdx.x; i < p.B; i += kThreads) sm.lens[i] = p.key_lens[i];
    if (warp == kLoadWarp && lane == 0) {
        prefetch_tensormap(&tmap_q);
        prefetch_tensormap(&tmap_k);
        prefetch_tensormap(&tmap_v);
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    {
        const int F = total / G, rem = total - F * G;
        if (threadIdx.x == 0) sm.n_items = F + ((((F & 1) ? (G - 1 - cta) : cta) < rem) ? 1 : 0);
        for (int t = threadIdx.x; t < kItemTable; t += kThreads) {
            const int k = item_index(t, cta, G);
            if (k < total) {
                const Item it = make_item(p, k, sm.lens);
                sm.item_tab[t][0] = it.bh;
                sm.item_tab[t][1] = it.b;
                sm.item_tab[t][2] = it.hh;
                sm.item_tab[t][3] = it.q0;
                sm.item_tab[t][4] = it.kv_len;
                sm.item_tab[t][5] = it.n_kv;
            }
        }
        __syncthreads();
    }
    const uint32_t tmem = sm.tmem_base;
    const AbortState ab{&sm.abort_flag, p.status, p.wait_limit_ns};
    // Programmatic dependent launch: the next kernel may begin its prologue;
    // nothing below touches global memory written by the kernel before this
    // one until that kernel has completed.
    pdl_launch_dependents();
    // Read the parameters every role needs for its first item now, while the
    // previous kernel drains: the first reads of the parameter block miss the
    // constant cache (~1,500 cycles measured at the start of each role).
    asm volatile("" ::"r"(p.B), "r"(p.H), "r"(p.Tq), "r"(p.Tk), "r"(p.num_qblocks), "r"(p.mask),
                 "r"(p.total_items), "f"(p.scale_log2), "l"(p.key_lens), "l"(p.o), "l"(p.status));
    pdl_wait();

    // Every role walks the same item list and counts, over the items that
    // have key tiles, the items (v: Q buffer v mod 2 and the per-item
    // barriers' phases) and the key tiles (g: stage g mod STAGES, score buffer
    // g mod 3).  Items without key tiles only produce zero rows.
    if (warp == kLoadWarp) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            int g = 0, v = 0;
            bool ok = true;
            for (int t = 0; ok; ++t) {
                if (t >= sm.n_items) break;
                const Item it = item_of(sm, p, t, cta, G);
                if (it.n_kv == 0) continue;
                const int qbuf = v & 1;
                // Q buffer qbuf last served item v-2: wait until all of its
                // score products have completed.
                if (v >= 2 && !(ok = mbar_wait(&sm.q_empty[qbuf], ((v - 2) >> 1) & 1, ab))) break;
                mbar_arrive_expect_tx(&sm.q_full[qbuf], kTileBytes);
                if (in_bounds(it.q0 >= 0 && it.q0 < p.Tq && it.bh >= 0 && it.bh < p.B * p.H, p.status))
                    tma_load_3d(&tmap_q, &sm.q_full[qbuf], sm.q[qbuf], 0, it.q0, it.bh);
                ++v;
                for (int j = 0; j < it.n_kv; ++j, ++g) {
                    const int st = g % STAGES;
                    if (g >= STAGES && !(ok = mbar_wait(&sm.kv_empty[st], ((g / STAGES) - 1) & 1, ab)))
                        break;
                    if (g + 1 == p.drill_skip_tile) continue;  // drill: this stage never fills
                    mbar_arrive_expect_tx(&sm.kv_full[st], 2 * kTileBytes);
                    if (in_bounds(j * BN < p.Tk && it.bh < p.B * p.H, p.status)) {
                        tma_load_3d(&tmap_k, &sm.kv_full[st], sm.k[st], 0, j * BN, it.bh);
                        tma_load_3d(&tmap_v, &sm.kv_full[st], sm.v[st], 0, j * BN, it.bh);
                    }
                }
            }
            // Let every copy still in flight land before the CTA exits (on the
            // normal path these phases completed long ago).
            for (int x = max(0, g - STAGES); x < g; ++x)
                if (x + 1 != p.drill_skip_tile) mbar_wait_drain(&sm.kv_full[x % STAGES], (x / STAGES) & 1);
            for (int x = max(0, v - 2); x < v; ++x) mbar_wait_drain(&sm.q_full[x & 1], (x >> 1) & 1);
        }
    } else if (warp == kMmaSWarp) {
        // ----------------------------------------------------- S issuer
        // S_g = Q K_g^T (4 MMAs, N = 128) into buffer g mod 3.  The whole
        // warp runs the loop and one elected lane issues (warp_mma_bf16_ss).
        // S_g overwrites the buffer of tile g-3, so it waits for the release
        // of tile g-3's stage (both P.V halves of tile g-3 complete; the
        // release of tile g-3+STAGES needs S_{g+2}, not yet issued, so the
        // parity cannot alias).
        constexpr uint32_t idesc_s = idesc_bf16_f32(BM, BN, false, false);
        // A K step of 16 adds 32 bytes (2 in the descriptor) in a K-major
        // row; a stage or Q buffer adds 16 KiB.
        constexpr uint64_t kTileDesc = kTileBytes >> 4;
        const uint64_t q_desc0 = smem_desc_sw128(smem_u32(sm.q[0]), 16, 1024);
        const uint64_t k_desc0 = smem_desc_sw128(smem_u32(sm.k[0]), 16, 1024);
        int g = 0, v = 0;
        bool ok = true;
        for (int t = 0; ok; ++t) {
            if (t >= sm.n_items) break;
            const Item it = item_of(sm, p, t, cta, G);
            if (it.n_kv == 0) continue;
            const int qbuf = v & 1;
            if (!(ok = warp_wait(&sm.q_full[qbuf], (v >> 1) & 1, ab))) break;
            const uint64_t qd = q_desc0 + static_cast<uint64_t>(qbuf) * kTileDesc;
            for (int j = 0; j < it.n_kv; ++j, ++g) {
                const int st = g % STAGES, sb = g % kSBufs;
                if (!(ok = warp_wait(&sm.kv_full[st], (g / STAGES) & 1, ab))) break;
                if (g >= kSBufs) {
                    const int gp = g - kSBufs;
                    if (!(ok = warp_wait(&sm.kv_empty[gp % STAGES], (gp / STAGES) & 1, ab))) break;
                }
                tc_fence_after_sync();
                const uint32_t d = tmem + 128u * static_cast<uint32_t>(sb);
                const uint64_t kd = k_desc0 + static_cast<uint64_t>(st) * kTileDesc;
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk)
                    warp_mma_bf16_ss(d, qd + 2 * kk, kd + 2 * kk, idesc_s, kk > 0 ? 1u : 0u);
                warp_commit(&sm.s_full[sb]);
            }
            if (!ok) break;
            // Every score product of this item is issued: the Q buffer is
            // free once they complete.
            warp_commit(&sm.q_empty[qbuf]);
            ++v;
        }
        // Always wait (time-bounded, whatever the abort state) until every
        // MMA this warp issued has completed: tensor memory is released and
        // the CTA exits only after that.
        warp_commit(&sm.drain[0]);
        mbar_wait_drain(&sm.drain[0], 0);
    } else if (warp == kMmaPvWarp || warp == kMmaPvWarp + 1) {
        // ---------------------------------------------------- PV issuers
        // Warp 10 + h: O_h (+)= P_g V_g for the tiles g with g mod 2 = h,
        // eight MMAs of 16 keys: A = P in tensor memory (8 columns per 16
        // keys, buffer columns [0,64)), B = V tile (MN-major, 16 keys = 2 KiB
        // = 128 per K step).  The group's first product of an item (j < 2)
        // overwrites O_h, so every item starts by waiting until the output
        // warps have read the previous item's accumulators; the item's
        // "output final" commit follows the group's last product (or none).
        const int hf = warp - kMmaPvWarp;
        constexpr uint32_t idesc_o = idesc_bf16_f32(BM, HD, false, true);
        constexpr uint64_t kTileDesc = kTileBytes >> 4;
        const uint64_t v_desc =
            smem_desc_sw128(smem_u32(sm.v[0]), 1024, 1024) + (kTiles ? 0 : 128 * 4 * hf);
        const uint32_t d_o = tmem + kOCol + 64u * static_cast<uint32_t>(hf);
        const uint32_t p_col = tmem + (kTiles ? 0u : 64u * static_cast<uint32_t>(hf));
        int g = 0, v = 0;
        bool ok = true;
        for (int t = 0; ok; ++t) {
            if (t >= sm.n_items) break;
            const Item it = item_of(sm, p, t, cta, G);
            if (it.n_kv == 0) continue;
            if (v >= 1 && !(ok = warp_wait(&sm.o_free, (v - 1) & 1, ab))) break;
            for (int j = 0; j < it.n_kv; ++j, ++g) {
                if (kTiles && (g & 1) != hf) continue;
                const int st = g % STAGES, sb = g % kSBufs;
                const int slot = (g >> 1) & 1, par = (g >> 2) & 1;
                if (!(ok = warp_wait(kTiles ? &sm.p_rd[hf][0][slot] : &sm.p_full[sb][hf],
                                     kTiles ? par : (g / kSBufs) & 1, ab)))
                    break;
                if (!(ok = warp_wait(&sm.kv_full[st], (g / STAGES) & 1, ab))) break;
                tc_fence_after_sync();
                const uint32_t a = p_col + 128u * static_cast<uint32_t>(sb);
                const uint64_t vd = v_desc + static_cast<uint64_t>(st) * kTileDesc;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    warp_mma_bf16_ts(d_o, a + 8 * kk, vd + 128 * kk, idesc_o,
                                     (j >= (kTiles ? 2 : 1) || kk > 0) ? 1u : 0u);
                if (kTiles) {
                    // The round-0 half is issued while the softmax works on
                    // round 1; the second half follows round 1's P.
                    warp_commit(&sm.pv0[hf][slot]);
                    if (!(ok = warp_wait(&sm.p_rd[hf][1][slot], par, ab))) break;
                    tc_fence_after_sync();
#pragma unroll
                    for (int kk = 4; kk < 8; ++kk)
                        warp_mma_bf16_ts(d_o, a + 8 * kk, vd + 128 * kk, idesc_o, 1u);
                }
                warp_commit(&sm.kv_empty[st]);
            }
            if (!ok) break;
            warp_commit(&sm.o_final);
            ++v;
        }
        warp_commit(&sm.drain[1 + hf]);
        mbar_wait_drain(&sm.drain[1 + hf], 0);
    } else if (warp < kSoftmaxWarps) {
        // --------------------------------------------------------- softmax
        // Group h owns the tiles g with g mod 2 = h, with its own reference
        // maximum m_h, running sum l_h and accumulator O_h; the two groups
        // are combined by the output warps.  A tile's 128 scores are taken
        // in two rounds of 64 (registers), each written back as 32 columns
        // of P over scores already read.
        //
        // Softmax is unchanged by a common shift of a row's scores, so P may
        // be taken against any reference m_h that keeps 2^(s c - m_h c)
        // finite; the running maximum is only one such choice.  A round is
        // therefore exponentiated straight against the current m_h (no
        // maximum pass), and the row checks its own round sum: only a row
        // whose sum exceeds 2^16 (its maximum grew by 10 to 16 log2 units or
        // more, or overflowed) takes the exact step -- round maximum, new
        // m_h, O_h and l_h scaled by 2^((m_old - m_new) c), P recomputed; in
        // the second round O_h is scaled once the first round's product is in
        // it.  Before the row has a reference its round is taken against 0
        // (any finite reference is valid) and kept when the sum lies in
        // [2^-64, 2^16] -- scores within about 16 log2 units of 0, as scaled
        // scores usually are; a sum outside (or no visible key, or an
        // exported lse) takes the exact step.  Each decision uses only the row's own visible scores,
        // so a row's result never depends on another row or on masked keys.
        const int half = warp >> 2;  // the group (by tiles) or key half (by halves)
        constexpr int kRounds = kTiles ? 2 : 1;  // 64-score rounds per tile
        const uint32_t lane_base = static_cast<uint32_t>(warp & 3) * 32;
        const int r = static_cast<int>(lane_base) + lane;    // row in tile = TMEM lane
        const uint32_t tl = tmem_addr(tmem, lane_base, 0);
        const uint32_t to = tl + kOCol + 64u * half;         // O_h: 64 columns
        const float C = p.scale_log2;
        // The first-round reference 0 only when no log-sum-exp is exported:
        // with the exact first step the row's largest weight is exactly 1,
        // so lse (and the weights a backward pass recomputes from it) carry
        // no rounding of that term.
        constexpr bool guess_first = !kLse;

        // Keys at or past `lim` (relative to the round's first key) get -inf:
        // weight exactly zero.
        auto mask_scores = [](uint32_t(&a)[32], uint32_t(&b)[32], int lim) {
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                if (c >= lim) a[c] = f2u(-INFINITY);
                if (c + 32 >= lim) b[c] = f2u(-INFINITY);
            }
        };
        // P = 2^(s c - mc) in bf16 (column c of the packed tile holds keys
        // 2c, 2c+1 of the round) and the fp32 row sum of P.  The sum adds
        // the bf16-rounded weights -- the values the P.V product multiplies
        // -- so numerator and denominator of the output carry the same
        // rounding and the normalised weights sum to 1: a key that dominates
        // its row returns its value row up to the output rounding, whatever
        // the reference maximum (with l summed from the unrounded weights
        // the output would be off by the relative rounding of the dominant
        // weight, up to 2^-8 |v|); the rounded weights are added by
        // mixed-precision adds (bf16 operand, fp32 sum), one instruction per
        // weight.  Packed fp32x2 FMA (one instruction per two scores) keeps
        // the instruction count -- and the issue slots taken from the MMA
        // warps -- down.
        auto exp_tile = [C](const uint32_t(&a)[32], const uint32_t(&b)[32], float mc,
                            uint32_t(&pk)[32]) -> float {
            const uint64_t c2 = f32x2_pack(C, C), nmc2 = f32x2_pack(-mc, -mc);
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                float x0, x1, x2, x3;
                f32x2_unpack(fma_f32x2(f32x2_pack(u2f(a[2 * c]), u2f(a[2 * c + 1])), c2, nmc2), x0, x1);
                f32x2_unpack(fma_f32x2(f32x2_pack(u2f(b[2 * c]), u2f(b[2 * c + 1])), c2, nmc2), x2, x3);
                pk[c] = pack_bf16x2(ex2_approx(x0), ex2_approx(x1));
                pk[16 + c] = pack_bf16x2(ex2_approx(x2), ex2_approx(x3));
                add_bf16x2_to_f32(acc[2 * (c & 1)], acc[2 * (c & 1) + 1], pk[c]);
                add_bf16x2_to_f32(acc[4 + 2 * (c & 1)], acc[5 + 2 * (c & 1)], pk[16 + c]);
            }
            return ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
        };
        // Row maximum of the round's 64 scores: four chains of three-input max.
        auto row_max = [](const uint32_t(&a)[32], const uint32_t(&b)[32]) -> float {
            float t0 = fmaxf(u2f(a[0]), u2f(a[1])), t1 = fmaxf(u2f(a[2]), u2f(a[3]));
            float t2 = fmaxf(u2f(b[0]), u2f(b[1])), t3 = fmaxf(u2f(b[2]), u2f(b[3]));
#pragma unroll
            for (int c = 4; c < 32; c += 4) {
                t0 = fmax3(t0, u2f(a[c]), u2f(a[c + 1]));
                t1 = fmax3(t1, u2f(a[c + 2]), u2f(a[c + 3]));
                t2 = fmax3(t2, u2f(b[c]), u2f(b[c + 1]));
                t3 = fmax3(t3, u2f(b[c + 2]), u2f(b[c + 3]));
            }
            return fmaxf(fmax3(t0, t1, t2), t3);
        };

        int g = 0, v = 0;
        bool ok = true;
        for (int t = 0; ok; ++t) {
            if (t >= sm.n_items) break;
            const Item it = item_of(sm, p, t, cta, G);
            if (it.n_kv == 0) continue;
            const int row = it.q0 + r;  // query index
            const int row_lim = causal ? min(it.kv_len, row + 1) : it.kv_len;  // keys < row_lim visible
            float m_run = -INFINITY;  // -inf until this group has seen a visible key
            float l_run = 0.f;

            for (int j = 0; j < it.n_kv; ++j, ++g) {
                if (kTiles && (g & 1) != half) continue;
                const int sb = g % kSBufs;
                ok = __all_sync(0xffffffffu, mbar_wait(&sm.s_full[sb], (g / kSBufs) & 1, ab));
                if (!ok) break;
                tc_fence_after_sync();
                const uint32_t ts = tl + 128u * static_cast<uint32_t>(sb);
                const bool edge =
                    (j * BN + BN > it.kv_len) || (causal && j * BN + BN - 1 > it.q0);
#pragma unroll
                for (int rd = 0; rd < kRounds; ++rd) {
                    const int c0 = kTiles ? 64 * rd : 64 * half;  // the round's first key in the tile
                    const uint32_t tr = ts + static_cast<uint32_t>(c0);
                    const int lim = row_lim - (j * BN + c0);
                    uint32_t pk[32];
                    float lt = 0.f;
                    bool need = true;  // no reference yet: exact unless the guess holds
                    if (guess_first || (kTiles ? (j >= 2 || rd == 1) : j > 0)) {
                        uint32_t s0[32], s1[32];
                        tmem_ld32(tr, s0);
                        tmem_ld32(tr + 32, s1);
                        tmem_ld_wait(s0);
                        reg_fence32(s1);
                        if (edge) mask_scores(s0, s1, lim);
                        lt = exp_tile(s0, s1, m_run == -INFINITY ? 0.f : m_run * C, pk);
                        // without a reference yet, the round was taken against 0:
                        // kept if its sum lies in [2^-64, 2^16], which then
                        // becomes the row's reference
                        need = m_run == -INFINITY
                                   ? !(guess_first && lt >= kFirstSumMin && lt <= kTileSumLimit)
                                   : !(lt <= kTileSumLimit);
                        if (!need && m_run == -INFINITY) m_run = 0.f;
                        // by halves (short items) a round with no visible key
                        // for this row -- the second key half of a diagonal
                        // tile -- has P = 0 exactly and needs no exact step (a
                        // missing reference stays missing)
                        if (!kTiles && lim <= 0) need = false;
                    }
                    if (__any_sync(0xffffffffu, need)) {
                        uint32_t s0[32], s1[32];
                        tmem_ld32(tr, s0);
                        tmem_ld32(tr + 32, s1);
                        tmem_ld_wait(s0);
                        reg_fence32(s1);
                        if (edge) mask_scores(s0, s1, lim);
                        float alpha = 1.f;
                        if (need) {
                            const float m_new = fmaxf(m_run, row_max(s0, s1));
                            if (m_run != -INFINITY) alpha = ex2_approx((m_run - m_new) * C);
                            m_run = m_new;
                            l_run *= alpha;
                            lt = exp_tile(s0, s1, m_run == -INFINITY ? 0.f : m_run * C, pk);
                        }
                        if (__any_sync(0xffffffffu, alpha != 1.f)) {
                            if (kTiles && rd == 1) {
                                // O_h holds the item's earlier tiles and this
                                // tile's round 0 (taken against the old
                                // reference): wait for that product.
                                ok = __all_sync(0xffffffffu, mbar_wait(&sm.pv0[half][(g >> 1) & 1],
                                                                       (g >> 2) & 1, ab));
                                if (!ok) break;
                                tc_fence_after_sync();
#pragma unroll 1
                                for (int part = 0; part < 2; ++part) {
                                    uint32_t o0[32];
                                    tmem_ld32(to + 32u * static_cast<uint32_t>(part), o0);
                                    tmem_ld_wait(o0);
#pragma unroll
                                    for (int c = 0; c < 32; ++c) o0[c] = f2u(u2f(o0[c]) * alpha);
                                    tmem_st32(to + 32u * static_cast<uint32_t>(part), o0);
                                    tmem_st_wait();
                                }
                            } else if (!kTiles || j >= 2) {
                                // O_h holds the earlier tiles of the item:
                                // wait for the product of the previous tile
                                // it took (g-2 by tiles; g-1, both halves, by
                                // halves, where a finite old reference means
                                // j >= 1).  That release's next phase needs
                                // P_g, not yet published, so it cannot alias.
                                const int gp = g - (kTiles ? 2 : 1);
                                ok = __all_sync(0xffffffffu,
                                                mbar_wait(&sm.kv_empty[gp % STAGES],
                                                          (gp / STAGES) & 1, ab));
                                if (!ok) break;
                                tc_fence_after_sync();
#pragma unroll 1
                                for (int part = 0; part < 2; ++part) {
                                    uint32_t o0[32];
                                    tmem_ld32(to + 32u * static_cast<uint32_t>(part), o0);
                                    tmem_ld_wait(o0);
#pragma unroll
                                    for (int c = 0; c < 32; ++c) o0[c] = f2u(u2f(o0[c]) * alpha);
                                    tmem_st32(to + 32u * static_cast<uint32_t>(part), o0);
                                    tmem_st_wait();
                                }
                            }

                        }
                    }
                    // P columns: [32 rd, 32 rd + 32) by tiles, [64 h, 64 h + 32)
                    // by halves; both lie over scores already read.
                    tmem_st32(ts + static_cast<uint32_t>(kTiles ? 32 * rd : 64 * half), pk);
                    l_run += lt;
                    if (kTiles) {
                        tmem_st_wait();
                        tc_fence_before_sync();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&sm.p_rd[half][rd][(g >> 1) & 1]);
                    }
                }
                if (!ok) break;
                if (!kTiles) {
                    tmem_st_wait();
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sm.p_full[sb][half]);
                }
            }
            if (!ok) break;
            // Row statistics of this item for the output warps, once they have
            // read the previous item's.
            if (v >= 1 && !(ok = __all_sync(0xffffffffu, mbar_wait(&sm.ml_free, (v - 1) & 1, ab))))
                break;
            sm.red_m[half][r] = m_run;
            sm.red_l[half][r] = l_run;
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.ml_full);
            ++v;
        }
        if (!ok) tmem_st_wait();  // no tensor-memory store may outlive the CTA
    } else if (warp >= kOutWarp) {
        // ------------------------------------------------------------ output
        // Warp 12 + q serves rows 32q .. 32q+31 (tensor-memory lane quadrant
        // q):
        //   out = (O_A w_A + O_B w_B) / (l_A w_A + l_B w_B),
        //   w_h = 2^((m_h - M) c), M = max(m_A, m_B);
        // a group that saw no visible key (or no tile) has weight 0 and its
        // accumulator, possibly never written for this item, is left out of
        // the result; a row with no visible key at all outputs 0.
        const uint32_t lane_base = static_cast<uint32_t>(warp & 3) * 32;
        const int r = static_cast<int>(lane_base) + lane;
        const uint32_t tl = tmem_addr(tmem, lane_base, 0);
        const float C = p.scale_log2;
        int v = 0;
        bool ok = true;
        for (int t = 0; ok; ++t) {
            if (t >= sm.n_items) break;
            const Item it = item_of(sm, p, t, cta, G);
            const int row = it.q0 + r;
            __nv_bfloat16 *dst = p.o + it.b * p.o_stride_b + it.hh * p.o_stride_h +
                                 static_cast<long long>(row) * p.o_stride_t;
            uint4 *d4 = reinterpret_cast<uint4 *>(dst);
            float *lse_row = p.lse && row < p.Tq
                                 ? p.lse + (static_cast<long long>(it.bh) * p.Tq + row)
                                 : nullptr;
            // The row's output lies inside the (B, H, T_q) index space.
            const bool row_ok = in_bounds(it.b < p.B && it.hh < p.H && row >= 0, p.status);
            if (!row_ok) lse_row = nullptr;
            if (it.n_kv == 0) {
                if (row < p.Tq && row_ok) {
#pragma unroll
                    for (int c = 0; c < 8; ++c) d4[c] = make_uint4(0u, 0u, 0u, 0u);
                    if (lse_row) *lse_row = -INFINITY;
                }
                continue;
            }
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(&sm.ml_full, v & 1, ab)))) break;
            const float ma = sm.red_m[0][r], mb = sm.red_m[1][r];
            const float la = sm.red_l[0][r], lb = sm.red_l[1][r];
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.ml_free);
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(&sm.o_final, v & 1, ab)))) break;
            tc_fence_after_sync();
            const float M = fmaxf(ma, mb);
            const float wa = la > 0.f ? ex2_approx((ma - M) * C) : 0.f;
            const float wb = lb > 0.f ? ex2_approx((mb - M) * C) : 0.f;
            const float L = la * wa + lb * wb;
            const float inv = L > 0.f ? 1.0f / L : 0.f;
            const float fa = wa * inv, fb = wb * inv;
            // Log-sum-exp of the row's visible scores: sum_j 2^(s_j c) =
            // 2^(M c) L with c = scale log2(e), so lse = M scale + ln L.
            // L sums the bf16-rounded weights (the normaliser of the output),
            // within a relative 2^-8 of the exact sum.
            if (lse_row) *lse_row = L > 0.f ? M * p.scale + logf(L) : -INFINITY;
#pragma unroll
            for (int part = 0; part < 2; ++part) {
                uint32_t oa[32], ob[32];
                tmem_ld32(tl + kOCol + 32u * part, oa);
                tmem_ld32(tl + kOCol + 64u + 32u * part, ob);
                tmem_ld_wait(oa);
                reg_fence32(ob);
                if (part == 1) {
                    // O_A and O_B are read: the next item's products may
                    // overwrite them.
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sm.o_free);
                }
                if (row < p.Tq && row_ok) {
                    uint32_t packed[16];
#pragma unroll
                    for (int c = 0; c < 16; ++c)
                        packed[c] = pack_bf16x2((la > 0.f ? u2f(oa[2 * c]) * fa : 0.f) +
                                                    (lb > 0.f ? u2f(ob[2 * c]) * fb : 0.f),
                                                (la > 0.f ? u2f(oa[2 * c + 1]) * fa : 0.f) +
                                                    (lb > 0.f ? u2f(ob[2 * c + 1]) * fb : 0.f));
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        d4[4 * part + c] = make_uint4(packed[4 * c], packed[4 * c + 1],
                                                      packed[4 * c + 2], packed[4 * c + 3]);
                }
            }
            ++v;
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == kMmaSWarp) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

bool attn_bf16_splits_by_tiles(int Tq, int Tk, int mask) {
    // Average key tiles per 128-row query tile (key padding ignored).
    const int nqb = (Tq + kAttnRowsPerCta - 1) / kAttnRowsPerCta;
    if (nqb <= 0 || Tk <= 0) return false;
    long long tiles = 0;
    for (int qb = 0; qb < nqb; ++qb) {
        const int kv_end = (mask & kMaskCausalBit) ? std::min(Tk, std::min((qb + 1) * kAttnRowsPerCta, Tq)) : Tk;
        tiles += (kv_end + BN - 1) / BN;
    }
    return tiles >= static_cast<long long>(kAttnTilesSplitMin) * nqb;
}

cudaError_t launch_attn_bf16(const CUtensorMap &tq, const CUtensorMap &tk,
                             const CUtensorMap &tv, const AttnParams &p, cudaStream_t stream,
                             bool pdl) {
    const bool by_tiles = attn_bf16_splits_by_tiles(p.Tq, p.Tk, p.mask);
    // kLse: the log-sum-exp is exported (the first round always exact)
    auto kernel = p.lse ? (by_tiles ? attn_fwd_bf16_kernel<true, true> : attn_fwd_bf16_kernel<false, true>)
                        : (by_tiles ? attn_fwd_bf16_kernel<true, false> : attn_fwd_bf16_kernel<false, false>);
    const size_t smem = sizeof(SmemAttn) + 1024;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    // One persistent CTA per SM (fewer if there are fewer items).
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return e;
    const int grid = p.total_items < sms ? p.total_items : sms;
    if (grid <= 0) return cudaSuccess;
    return launch_kernel(kernel, dim3(grid), dim3(kThreads), smem, stream, pdl, 1, tq, tk, tv, p);
}

}  // namespace mha
