// The post-mix of one layer fused with the projection pass of the next
// (cross-op fusion: h_post_bda of layer l, whose output is the residual
// input of layer l+1, and the sum-of-squares / thin-projection pass of
// proj_rms_compute_h on that input; RL-Kernel PR #383 names fusing
// fp32_gemm_rms with its producer, Megatron-Core fused_mhc_kernels the two
// ops).  Per token t:
//   out[t][i][c] = sum_j H_res[t][j][i] x[t][j][c] + H_post[t][i] (f[t][c] + bias[c])   (bf16)
//   upart[s][t][o] = sum_{k in s} out[t][k] W'[k][o],  spart[s][t] = sum_{k in s} out[t][k]^2
// with k = i*C + c and out taken as stored (bf16), so the next layer sees
// exactly what a separate projection pass over `out` would read.  The
// partial sums then go through the usual compute_h (next layer's H).
//
// n = 4.  CTA: 128 tokens x a range of channel blocks; a stage is one
// channel block of BC channels: the n residual boxes [128 x BC] and f's box
// (TMA, swizzled) plus the n W'_hl boxes [NB x BC] of its k-blocks (W' as
// three bf16 terms hi | lo | lo2 and zero rows, NB = 80).  Warps:
//   0     TMA producer
//   1     TMEM, then per stage: TMA store of the stage's out boxes to HBM and
//         the MMAs out . [W'_lo | W'_lo2] (N = 48, accumulated over the split)
//         and out . W'_hi (N = 32) into one of two buffers per group of G
//         stages, which the epilogue warps drain into fp32 registers (the
//         tensor core's accumulator loses about an ulp of the running sum per
//         K step, so the large term is not accumulated over the split)
//   2..9  two warps per token row r (half the block's channels each): out for the row's
//         channels of every stream, written over the residual boxes in place
//         (same swizzled layout, so the boxes become both the MMA A operand
//         and the store source); the row's sum of squares of the bf16
//         outputs; at the end of each group the first warp of a quadrant
//         drains its out . W'_hi buffer; finally TMEM -> partials
// A stage is free again when its MMAs have completed and the store has read
// it.  Channels past C and rows past T load as zeros and are not stored.
#include "launch.h"
#include "tc.cuh"
#include "tmap.h"

#include <cstring>

namespace mhc {

// BC channels per stage (64: 128-byte rows and swizzle; 32: 64-byte rows
// and swizzle), STAGES stages, MINB CTAs per SM.
template <int BC_, int STAGES_, int MINB_>
struct PostProjCfg {
    static constexpr int N = 4, O = N * N + 2 * N, NB = w_split_rows(4);  // 24 logits, 80 MMA columns
    static constexpr int BM = 128, BC = BC_;                     // tokens, channels per stage
    static constexpr int RB = BC * 2;                            // bytes of a box row
    static constexpr int CH = BC / 8;                            // 16-byte chunks per row
    static constexpr int XBOX = BM * RB;                         // one stream's box
    static constexpr int F_OFF = N * XBOX;
    static constexpr int WBOX = NB * RB;
    static constexpr int W_OFF = F_OFF + XBOX;
    static constexpr int STAGE = W_OFF + N * WBOX;
    static constexpr int STAGES = STAGES_, MINB = MINB_;
    static constexpr int SMEM = STAGES * STAGE + 1024;
    // TMEM: two out.W'_hi buffers (NH = 32 columns, 24 used) and the
    // [out.W'_lo | out.W'_lo2] accumulator (NL = 48), drained every G stages
    static constexpr int NH = 32, NL = 2 * O, HI0 = 0, HI1 = NH, LO = 2 * NH, G = 2;
    static constexpr int TMEM_COLS = 128;
    static_assert(LO + NL <= TMEM_COLS && 3 * O <= NB, "accumulators");
    static constexpr int WORKERS = 8;  // warps 2..9
    static constexpr int THREADS = 64 + 32 * WORKERS;
    static constexpr int ATOM = BC == 64 ? 1024 : 512;  // swizzle pattern repeat
    static_assert(BC == 64 || BC == 32, "box width");
    static_assert(XBOX % ATOM == 0 && WBOX % ATOM == 0 && STAGE % 1024 == 0, "alignment");
    static_assert((SMEM + 1024) * MINB <= 233472, "shared memory");
    // 16-byte chunk cc of row r in the swizzled box
    __device__ static uint32_t chunk_off(int r, int cc)
    {
        return uint32_t(r * RB + ((BC == 64 ? (cc ^ (r & 7)) : (cc ^ ((r >> 1) & 3))) << 4));
    }
    __device__ static uint64_t desc(uint32_t addr)
    {
        return BC == 64 ? tc::desc_kmajor_sw128(addr) : tc::make_desc(addr, 16, 512, tc::kSwz64);
    }
};
// Three 60 KB stages of 32 channels, one CTA per SM.  (With W' in two terms,
// 52 KB stages: four stages 0.217 ms at T=16384, n=4, C=4096; two 104 KB
// stages of 64 channels 0.244 ms; two stages at two CTAs per SM 0.248 ms.)
using PostProj = PostProjCfg<32, 3, 1>;

template <class P>
__global__ void __launch_bounds__(P::THREADS, P::MINB)
    k_post_proj_tc(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmf,
                   const __grid_constant__ CUtensorMap tmo, const bf16 *__restrict__ Wt,
                   const bf16 *__restrict__ bias, const float *__restrict__ Hres,
                   const float *__restrict__ Hpost, float *__restrict__ upart,
                   float *__restrict__ spart, int64_t T, int64_t C, int cb_per_split,
                   int cb_total, int *fault)
{
    pdl_wait();
    constexpr int N = P::N, O = P::O;
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t full[P::STAGES], ready[P::STAGES], empty[P::STAGES], acc_bar, hifull[2],
        hiempty[2];
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    __shared__ float ssq_red[P::BM];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    volatile int *abort_v = &abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = int(blockIdx.x) * P::BM;
    const int split = int(blockIdx.y);
    const int cb0 = split * cb_per_split;
    const int ncb = min(cb_total, cb0 + cb_per_split) - cb0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < P::STAGES; ++s) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&ready[s], 32 * P::WORKERS);  // every worker thread
            tc::mbar_init(&empty[s], 2);  // the MMAs' commit + the store's read
        }
        tc::mbar_init(&acc_bar, 1);
        for (int hb = 0; hb < 2; ++hb) {
            tc::mbar_init(&hifull[hb], 1);
            tc::mbar_init(&hiempty[hb], 4);   // the first worker warp of each quadrant
        }
        abort_flag = 0;
        tc::fence_barrier_init();
    }
    if (warp == 1) tc::tmem_alloc(&tmem_slot, P::TMEM_COLS);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            tc::tma_prefetch_desc(&tmx);
            tc::tma_prefetch_desc(&tmf);
            int issued = 0;
            for (int i = 0; i < ncb && !*abort_v; ++i) {
                const int s = i % P::STAGES;
                if (i >= P::STAGES &&
                    !tc::mbar_wait(&empty[s], ((i / P::STAGES) & 1) ^ 1, fault,
                                   tc::kFaultTimeoutEmpty)) {
                    *abort_v = 1;
                    break;
                }
                uint8_t *st = smem + s * P::STAGE;
                const int c0 = (cb0 + i) * P::BC;
                tc::mbar_arrive_expect_tx(&full[s], P::STAGE);
                for (int j = 0; j < N; ++j) tc::tma_load_3d(st + j * P::XBOX, &tmx, c0, j, m0, &full[s]);
                tc::tma_load_2d(st + P::F_OFF, &tmf, c0, m0, &full[s]);
                // the block's W stage is one contiguous image (k_w_tile)
                tc::bulk_load(st + P::W_OFF,
                              reinterpret_cast<const uint8_t *>(Wt) + int64_t(cb0 + i) * N * P::WBOX,
                              N * P::WBOX, &full[s]);
                issued = i + 1;
            }
            // do not leave while copies into this CTA's shared memory are in flight
            for (int i = max(0, issued - P::STAGES); i < issued; ++i)
                tc::mbar_wait(&full[i % P::STAGES], (i / P::STAGES) & 1, fault,
                              tc::kFaultTimeoutMisc);
        }
    } else if (warp == 1) {
        // ------------------------------------------------- out store + MMA issue
        if (lane == 0) {
            tc::tma_prefetch_desc(&tmo);
            constexpr uint32_t idesc_hi = tc::idesc_bf16_f32(P::BM, P::NH);
            constexpr uint32_t idesc_lo = tc::idesc_bf16_f32(P::BM, P::NL);
            bool ok = true;
            for (int i = 0; i < ncb; ++i) {
                const int s = i % P::STAGES, g = i / P::G, hb = g & 1;
                const bool first = i % P::G == 0, last = i % P::G == P::G - 1 || i == ncb - 1;
                if (*abort_v ||
                    !tc::mbar_wait(&ready[s], (i / P::STAGES) & 1, fault, tc::kFaultTimeoutFull)) {
                    ok = false;
                    break;
                }
                tc::tc_fence_after();
                uint8_t *st = smem + s * P::STAGE;
                const int c0 = (cb0 + i) * P::BC;
                for (int j = 0; j < N; ++j) tc::tma_store_3d(&tmo, st + j * P::XBOX, c0, j, m0);
                tc::bulk_commit_group();
                const uint32_t a0 = tc::smem_u32(st);
                // W'_hl rows [O, 3O) (lo | lo2) start on an 8-row swizzle group
#pragma unroll
                for (int j = 0; j < N; ++j) {
                    const uint32_t a = a0 + j * P::XBOX, b = a0 + P::W_OFF + j * P::WBOX;
#pragma unroll
                    for (int kk = 0; kk < P::BC / 16; ++kk)
                        tc::mma_bf16(tmem + P::LO, P::desc(a + kk * 32),
                                     P::desc(b + O * P::RB + kk * 32), idesc_lo,
                                     (i > 0 || j > 0 || kk > 0) ? 1u : 0u);
                }
                // the out.W'_hi buffer must have been drained (group g - 2)
                if (first && g >= 2 &&
                    !tc::mbar_wait(&hiempty[hb], ((g >> 1) - 1) & 1, fault, tc::kFaultTimeoutAcc)) {
                    ok = false;
                    break;
                }
                tc::tc_fence_after();
#pragma unroll
                for (int j = 0; j < N; ++j) {
                    const uint32_t a = a0 + j * P::XBOX, b = a0 + P::W_OFF + j * P::WBOX;
#pragma unroll
                    for (int kk = 0; kk < P::BC / 16; ++kk)
                        tc::mma_bf16(tmem + (hb ? P::HI1 : P::HI0), P::desc(a + kk * 32),
                                     P::desc(b + kk * 32), idesc_hi,
                                     (!first || j > 0 || kk > 0) ? 1u : 0u);
                }
                tc::mma_commit(&empty[s]);
                if (last) tc::mma_commit(&hifull[hb]);
                tc::bulk_wait_read_all();
                tc::mbar_arrive(&empty[s]);
            }
            if (!ok) *abort_v = 1;
            tc::mma_commit(&acc_bar);
            tc::mbar_wait(&acc_bar, 0, fault, tc::kFaultTimeoutAcc);
            tc::bulk_wait_all();
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ workers
        // two warps per TMEM lane quadrant; warp half `hf` takes half of the
        // 16-byte chunks of every row of the quadrant
        const int q = warp & 3;
        const int hf = (warp - 2) >> 2;
        const int r = q * 32 + lane;  // token row of the tile = TMEM lane
        const int64_t t = int64_t(m0) + r;
        const bool live = t < T;
        // the row's H_res and H_post as f32x2 pairs (the same value twice)
        f32x2 hr2[N * N], hp2[N];
#pragma unroll
        for (int e = 0; e < N * N; e += 4) {
            const float4 v = live ? __ldg(reinterpret_cast<const float4 *>(Hres + t * N * N + e))
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
            hr2[e] = f2_make(v.x, v.x);
            hr2[e + 1] = f2_make(v.y, v.y);
            hr2[e + 2] = f2_make(v.z, v.z);
            hr2[e + 3] = f2_make(v.w, v.w);
        }
        {
            const float4 v = live ? __ldg(reinterpret_cast<const float4 *>(Hpost + t * N))
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
            hp2[0] = f2_make(v.x, v.x);
            hp2[1] = f2_make(v.y, v.y);
            hp2[2] = f2_make(v.z, v.z);
            hp2[3] = f2_make(v.w, v.w);
        }
        f32x2 ssq2 = 0ull;
        const uint32_t trow = tmem + (uint32_t(q * 32) << 16);
        float uhi[O];   // (hf = 0) sum over the groups of out.W'_hi, fp32 round to nearest
#pragma unroll
        for (int o = 0; o < O; ++o) uhi[o] = 0.f;
        bool ok = true;
        for (int i = 0; i < ncb; ++i) {
            const int s = i % P::STAGES;
            if (*abort_v ||
                !tc::mbar_wait(&full[s], (i / P::STAGES) & 1, fault, tc::kFaultTimeoutFull)) {
                *abort_v = 1;
                ok = false;
                break;
            }
            const uint32_t st = tc::smem_u32(smem + s * P::STAGE);
            const int c0 = (cb0 + i) * P::BC;
#pragma unroll 2
            for (int c4 = 0; c4 < P::CH / 2; ++c4) {
                const int cc = (P::CH / 2) * hf + c4;
                const uint32_t off = P::chunk_off(r, cc);
                const int64_t c = int64_t(c0) + cc * 8;
                f32x2 fb[4], bb[4];
                unpack8x2(lds128(st + P::F_OFF + off), fb);
                unpack8x2((bias && c < C) ? __ldg(reinterpret_cast<const uint4 *>(bias + c))
                                          : make_uint4(0, 0, 0, 0),
                          bb);
#pragma unroll
                for (int e = 0; e < 4; ++e) fb[e] = f2_add(fb[e], bb[e]);
                // the same fp32 operations per element as the separate
                // post-mix: H_post (f + bias), then H_res[j][i] x_j for j ascending
                f32x2 acc[N][4];
#pragma unroll
                for (int ii = 0; ii < N; ++ii)
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[ii][e] = f2_mul(hp2[ii], fb[e]);
#pragma unroll
                for (int j = 0; j < N; ++j) {
                    f32x2 v[4];
                    unpack8x2(lds128(st + j * P::XBOX + off), v);
#pragma unroll
                    for (int ii = 0; ii < N; ++ii)
#pragma unroll
                        for (int e = 0; e < 4; ++e) acc[ii][e] = f2_fma(hr2[j * N + ii], v[e], acc[ii][e]);
                }
                // out stream ii replaces residual stream ii in place
#pragma unroll
                for (int ii = 0; ii < N; ++ii) {
                    const uint4 o = pack8x2(acc[ii]);
                    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(st + ii * P::XBOX + off),
                                 "r"(o.x), "r"(o.y), "r"(o.z), "r"(o.w)
                                 : "memory");
                    f32x2 rv[4];
                    unpack8x2(o, rv);
#pragma unroll
                    for (int e = 0; e < 4; ++e) ssq2 = f2_fma(rv[e], rv[e], ssq2);
                }
            }
            // the out boxes are read by the tensor cores and the TMA store:
            // each thread's writes are complete before its arrival
            tc::fence_proxy_async_smem();
            tc::mbar_release(&ready[s]);
            // end of a group: the first warp of the quadrant drains its rows'
            // out.W'_hi buffer into registers and hands it back
            const int g = i / P::G, hb = g & 1;
            if (hf == 0 && (i % P::G == P::G - 1 || i == ncb - 1)) {
                if (*abort_v ||
                    !tc::mbar_wait(&hifull[hb], (g >> 1) & 1, fault, tc::kFaultTimeoutAcc)) {
                    *abort_v = 1;
                    ok = false;
                    break;
                }
                tc::tc_fence_after();
                float w0[16], w1[16];
                tc::tmem_ld16x2_wait(trow + (hb ? P::HI1 : P::HI0), trow + (hb ? P::HI1 : P::HI0) + 16,
                                     w0, w1);
#pragma unroll
                for (int e = 0; e < 16; ++e) uhi[e] += w0[e];
#pragma unroll
                for (int e = 0; e < O - 16; ++e) uhi[16 + e] += w1[e];
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&hiempty[hb]);
            }
        }
        float s_lo, s_hi;
        f2_split(ssq2, s_lo, s_hi);
        const float ssq = s_lo + s_hi;
        // the row's sum of squares: half 1 hands its part to half 0
        if (hf == 1) ssq_red[r] = ssq;
        tc::named_bar_sync(1 + q, 64);
        if (hf == 0) {
            const float ssq_row = ssq + ssq_red[r];
            if (ok && !tc::mbar_wait(&acc_bar, 0, fault, tc::kFaultTimeoutAcc)) ok = false;
            tc::tc_fence_after();
            // u = sum over groups of out.W'_hi + (out.W'_lo + out.W'_lo2)
#pragma unroll
            for (int c = 0; c < O / 8; ++c) {
                float w[8], w2[8];
                tc::tmem_ld8x2_wait(trow + P::LO + c * 8, trow + P::LO + O + c * 8, w, w2);
#pragma unroll
                for (int e = 0; e < 8; ++e) uhi[c * 8 + e] += w[e] + w2[e];
            }
            if (ok && !*abort_v && live) {
                float4 *dst = reinterpret_cast<float4 *>(upart + (int64_t(split) * T + t) * O);
#pragma unroll
                for (int o4 = 0; o4 < O / 4; ++o4)
                    dst[o4] = make_float4(uhi[4 * o4], uhi[4 * o4 + 1], uhi[4 * o4 + 2], uhi[4 * o4 + 3]);
                spart[int64_t(split) * T + t] = ssq_row;
            }
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) tc::tmem_dealloc(tmem, P::TMEM_COLS);
}

// ---------------------------------------------------------------------------
// n = 8.  The same dataflow with 16-channel stages: the 8 residual boxes
// [128 x 16] and f's box (32-byte rows, 32-byte swizzle) and the 8 W'_hl
// boxes [240 x 16] of the block's k-blocks (96 KB, two stages).  Each worker
// thread owns one token row and one 8-channel half of the block and forms
// all 8 output streams of it; the row's H_res and H_post sit in registers as
// pairs of neighbouring outputs, so the mix runs in paired fp32 operations
// (fma.rn.f32x2: per element the same single-rounding fmaf, in the same
// order as the separate post-mix).  Per stage and output stream:
// out.[W'_lo | W'_lo2] (N = 160, accumulated over the split) and out.W'_hi
// (N = 80) into one of two buffers drained every G stages into an fp32 sum
// kept in spare TMEM columns (both worker warps of a quadrant drain half of
// the 80 columns).
// ---------------------------------------------------------------------------
struct PostProj8 {
    static constexpr int N = 8, O = N * N + 2 * N, NB = w_split_rows(8);  // 80 logits, 240 rows
    static constexpr int BM = 128, BC = 16, RB = BC * 2;                  // 32-byte box rows
    static constexpr int XBOX = BM * RB;                                  // 4 KB
    static constexpr int XSTAGE = N * XBOX;                               // 32 KB
    static constexpr int WBOX = NB * RB;                                  // 7.5 KB
    static constexpr int WSTAGE = N * WBOX;                               // 60 KB
    static constexpr int XSTAGES = 3, WSTAGES = 2;
    // x and f are also prefetched into L2 in boxes of PF_C channels (64-byte
    // rows: a stage's own 32-byte rows, 14 KB apart, make poor DRAM bursts),
    // PF_AHEAD stages ahead of the loads.  Measured at T = 8192, C = 7168:
    // 32 channels 2 stages ahead 0.522 ms; 64 channels 4 ahead 0.530; none
    // 0.545; 64 channels 8 ahead 0.579 and 128 channels 8 ahead 0.581 (what
    // is prefetched that far ahead is evicted by the streaming out stores
    // before use and read again: 623 MB of DRAM reads for 292 MB of inputs)
    static constexpr int PF_C = 32, PF_STAGES = PF_C / BC, PF_AHEAD = 2;
    static constexpr int W_OFF = XSTAGES * XSTAGE;
    static constexpr int B_OFF = W_OFF + WSTAGES * WSTAGE;                // bias[16] per x stage,
    static constexpr int BSLOT = 128;                                     // TMA destinations 128-byte aligned
    static constexpr int SMEM = B_OFF + XSTAGES * BSLOT + 1024;
    static constexpr int NH = O, NL = 2 * O, HI0 = 0, HI1 = NH, LO = 2 * NH, UACC = LO + NL, G = 2;
    static constexpr int TMEM_COLS = 512;
    static constexpr int WORKERS = 8;
    static constexpr int THREADS = 64 + 32 * WORKERS;
    static_assert(UACC + O <= TMEM_COLS && 3 * O == NB, "TMEM columns");
    static_assert(XSTAGE % 1024 == 0 && WSTAGE % 1024 == 0 && XBOX % 256 == 0 && WBOX % 256 == 0 &&
                      W_OFF % 1024 == 0 && B_OFF % 128 == 0,
                  "alignment");
    static_assert(SMEM + 1024 <= 232448, "shared memory");
    // 16-byte chunk cc (0 or 1) of row r in the 32-byte swizzle
    __device__ static uint32_t chunk_off(int r, int cc) { return uint32_t(r * RB + ((cc ^ ((r >> 2) & 1)) << 4)); }
    __device__ static uint64_t desc(uint32_t addr) { return tc::make_desc(addr, 16, 256, tc::kSwz32); }
};

__global__ void __launch_bounds__(PostProj8::THREADS, 1)
    k_post_proj8_tc(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmb,
                    const __grid_constant__ CUtensorMap tmo, const __grid_constant__ CUtensorMap tmxp,
                    const __grid_constant__ CUtensorMap tmfp, const bf16 *__restrict__ Wt,
                    const bf16 *__restrict__ f, const bf16 *__restrict__ bias,
                    const float *__restrict__ Hres, const float *__restrict__ Hpost,
                    float *__restrict__ upart, float *__restrict__ spart, int64_t T, int64_t C,
                    int cb_per_split, int cb_total, int *fault)
{
    pdl_wait();
    using P = PostProj8;
    constexpr int N = P::N, O = P::O, XS = P::XSTAGES, WS = P::WSTAGES;
    extern __shared__ uint8_t smem_raw[];
    // x stages: full (TMA) -> ready (workers wrote out) -> empty (MMAs done and
    // the store has read them); W stages: wfull (TMA) -> wempty (MMAs done)
    __shared__ uint64_t full[XS], ready[XS], empty[XS], wfull[WS], wempty[WS], acc_bar, hifull[2],
        hiempty[2];
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    __shared__ float ssq_red[P::BM];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    volatile int *abort_v = &abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = int(blockIdx.x) * P::BM;
    const int split = int(blockIdx.y);
    const int cb0 = split * cb_per_split;
    const int ncb = min(cb_total, cb0 + cb_per_split) - cb0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < XS; ++s) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&ready[s], 32 * P::WORKERS);   // every worker thread
            tc::mbar_init(&empty[s], 2);                 // the MMAs' commit + the store's read
        }
        for (int s = 0; s < WS; ++s) {
            tc::mbar_init(&wfull[s], 1);
            tc::mbar_init(&wempty[s], 1);
        }
        tc::mbar_init(&acc_bar, 1);
        for (int hb = 0; hb < 2; ++hb) {
            tc::mbar_init(&hifull[hb], 1);
            tc::mbar_init(&hiempty[hb], P::WORKERS);
        }
        abort_flag = 0;
        tc::fence_barrier_init();
    }
    if (warp == 1) tc::tmem_alloc(&tmem_slot, P::TMEM_COLS);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            tc::tma_prefetch_desc(&tmx);
            if (bias) tc::tma_prefetch_desc(&tmb);
            int issued = 0, wissued = 0;
            // L2 prefetch of the PF_C-channel group holding stage i (i a multiple of PF_STAGES)
            auto prefetch = [&](int i) {
                if (i >= ncb) return;
                const int c = (cb0 + i) * P::BC;
                for (int j = 0; j < N; ++j) tc::tma_prefetch_l2_3d(&tmxp, c, j, m0);
                tc::tma_prefetch_l2_2d(&tmfp, c, m0);
            };
            for (int i = 0; i < P::PF_AHEAD; i += P::PF_STAGES) prefetch(i);
            for (int i = 0; i < ncb && !*abort_v; ++i) {
                const int xs = i % XS, ws = i % WS;
                const int c0 = (cb0 + i) * P::BC;
                if (i % P::PF_STAGES == 0) prefetch(i + P::PF_AHEAD);
                if (i >= XS && !tc::mbar_wait(&empty[xs], ((i / XS) & 1) ^ 1, fault,
                                              tc::kFaultTimeoutEmpty)) {
                    *abort_v = 1;
                    break;
                }
                uint8_t *st = smem + xs * P::XSTAGE;
                tc::mbar_arrive_expect_tx(&full[xs], P::XSTAGE + (bias ? P::RB : 0));
                for (int j = 0; j < N; ++j) tc::tma_load_3d(st + j * P::XBOX, &tmx, c0, j, m0, &full[xs]);
                if (bias) tc::tma_load_2d(smem + P::B_OFF + xs * P::BSLOT, &tmb, c0, 0, &full[xs]);
                issued = i + 1;
                if (i >= WS && !tc::mbar_wait(&wempty[ws], ((i / WS) & 1) ^ 1, fault,
                                              tc::kFaultTimeoutEmpty)) {
                    *abort_v = 1;
                    break;
                }
                // the block's W stage is one contiguous image (k_w_tile8)
                tc::mbar_arrive_expect_tx(&wfull[ws], P::WSTAGE);
                tc::bulk_load(smem + P::W_OFF + ws * P::WSTAGE,
                              reinterpret_cast<const uint8_t *>(Wt) + int64_t(cb0 + i) * P::WSTAGE,
                              P::WSTAGE, &wfull[ws]);
                wissued = i + 1;
            }
            // the last loads land before the CTA can exit
            for (int i = max(0, issued - XS); i < issued; ++i)
                tc::mbar_wait(&full[i % XS], (i / XS) & 1, fault, tc::kFaultTimeoutMisc);
            for (int i = max(0, wissued - WS); i < wissued; ++i)
                tc::mbar_wait(&wfull[i % WS], (i / WS) & 1, fault, tc::kFaultTimeoutMisc);
        }
    } else if (warp == 1) {
        // ------------------------------------------------- out store + MMA issue
        if (lane == 0) {
            tc::tma_prefetch_desc(&tmo);
            constexpr uint32_t idesc_hi = tc::idesc_bf16_f32(P::BM, P::NH);
            constexpr uint32_t idesc_lo = tc::idesc_bf16_f32(P::BM, P::NL);
            bool ok = true;
            for (int i = 0; i < ncb; ++i) {
                const int xs = i % XS, ws = i % WS, g = i / P::G, hb = g & 1;
                const bool first = i % P::G == 0, last = i % P::G == P::G - 1 || i == ncb - 1;
                if (*abort_v ||
                    !tc::mbar_wait(&ready[xs], (i / XS) & 1, fault, tc::kFaultTimeoutFull) ||
                    !tc::mbar_wait(&wfull[ws], (i / WS) & 1, fault, tc::kFaultTimeoutFull)) {
                    ok = false;
                    break;
                }
                tc::tc_fence_after();
                uint8_t *st = smem + xs * P::XSTAGE;
                const int c0 = (cb0 + i) * P::BC;
                const uint32_t a0 = tc::smem_u32(st);
                const uint32_t b0 = tc::smem_u32(smem + P::W_OFF + ws * P::WSTAGE);
                // W'_hl rows [80, 240) (lo | lo2): 80 rows = ten 8-row swizzle groups
#pragma unroll
                for (int j = 0; j < N; ++j)
                    tc::mma_bf16(tmem + P::LO, P::desc(a0 + j * P::XBOX),
                                 P::desc(b0 + j * P::WBOX + O * P::RB), idesc_lo,
                                 (i > 0 || j > 0) ? 1u : 0u);
                if (first && g >= 2 &&
                    !tc::mbar_wait(&hiempty[hb], ((g >> 1) - 1) & 1, fault, tc::kFaultTimeoutAcc)) {
                    ok = false;
                    break;
                }
                tc::tc_fence_after();
#pragma unroll
                for (int j = 0; j < N; ++j)
                    tc::mma_bf16(tmem + (hb ? P::HI1 : P::HI0), P::desc(a0 + j * P::XBOX),
                                 P::desc(b0 + j * P::WBOX), idesc_hi, (!first || j > 0) ? 1u : 0u);
                tc::mma_commit(&empty[xs]);
                tc::mma_commit(&wempty[ws]);
                if (last) tc::mma_commit(&hifull[hb]);
                // the store after the MMAs: its issue can wait behind queued loads
                for (int j = 0; j < N; ++j) tc::tma_store_3d(&tmo, st + j * P::XBOX, c0, j, m0);
                tc::bulk_commit_group();
                tc::bulk_wait_read_all();
                tc::mbar_arrive(&empty[xs]);
            }
            if (!ok) *abort_v = 1;
            tc::mma_commit(&acc_bar);
            tc::mbar_wait(&acc_bar, 0, fault, tc::kFaultTimeoutAcc);
            tc::bulk_wait_all();
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ workers
        const int q = warp & 3;
        const int hf = (warp - 2) >> 2;       // this warp's 8-channel half of the block
        const int r = q * 32 + lane;          // token row = TMEM lane
        const int64_t t = int64_t(m0) + r;
        const bool live = t < T;
        const uint32_t trow = tmem + (uint32_t(q * 32) << 16);
        // hw[j][k] = (H_res[t][j][2k], H_res[t][j][2k+1]), hq[k] = (H_post[t][2k], H_post[t][2k+1])
        f32x2 hw[N][N / 2], hq[N / 2];
#pragma unroll
        for (int j = 0; j < N; ++j)
#pragma unroll
            for (int k = 0; k < N / 2; ++k) {
                const float2 h = live ? __ldg(reinterpret_cast<const float2 *>(Hres + (t * N + j) * N) + k)
                                      : make_float2(0.f, 0.f);
                hw[j][k] = f2_make(h.x, h.y);
            }
#pragma unroll
        for (int k = 0; k < N / 2; ++k) {
            const float2 h = live ? __ldg(reinterpret_cast<const float2 *>(Hpost + t * N) + k)
                                  : make_float2(0.f, 0.f);
            hq[k] = f2_make(h.x, h.y);
        }
        constexpr int OH = O / 2;   // this warp's half of the logits: [hf OH, hf OH + OH)
        const uint32_t ucol = trow + P::UACC + hf * OH;
        f32x2 ssq2 = f2_make(0.f, 0.f);
        bool ok = true;
        // f's chunk of the row is read from global memory one stage ahead
        const bf16 *frow = f + t * C + hf * 8;
        auto load_f = [&](int i) {
            const int64_t c = int64_t(cb0 + i) * P::BC;
            return (live && i < ncb && c + hf * 8 < C) ? __ldg(reinterpret_cast<const uint4 *>(frow + c)) : make_uint4(0, 0, 0, 0);
        };
        uint4 fnext = load_f(0);
        for (int i = 0; i < ncb; ++i) {
            const int s = i % XS;
            const uint4 fcur = fnext;
            fnext = load_f(i + 1);
            if (*abort_v ||
                !tc::mbar_wait(&full[s], (i / XS) & 1, fault, tc::kFaultTimeoutFull)) {
                *abort_v = 1;
                ok = false;
                break;
            }
            const uint32_t st = tc::smem_u32(smem + s * P::XSTAGE);
            const uint32_t off = P::chunk_off(r, hf);
            // the same fp32 operations per element as the separate post-mix:
            // fb = f + bias, H_post[i] fb, then fmaf(H_res[j][i], x_j, .) for j ascending
            // (bias channels past C load as zeros)
            float fb[8], bb[8];
            unpack8(fcur, fb);
            unpack8(bias ? lds128(tc::smem_u32(smem + P::B_OFF + s * P::BSLOT) + hf * 16)
                         : make_uint4(0, 0, 0, 0),
                    bb);
#pragma unroll
            for (int e = 0; e < 8; ++e) fb[e] += bb[e];
            // four channels at a time (8-byte shared accesses, two-way bank
            // conflicts: the same wavefronts as conflict-free 16-byte ones)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                f32x2 acc[N / 2][4];   // acc[k][e]: outputs 2k, 2k+1 at channel 4h + e
#pragma unroll
                for (int e = 0; e < 4; ++e)
#pragma unroll
                    for (int k = 0; k < N / 2; ++k)
                        acc[k][e] = f2_mul(hq[k], f2_make(fb[4 * h + e], fb[4 * h + e]));
#pragma unroll
                for (int j = 0; j < N; ++j) {
                    const uint2 w = lds64(st + j * P::XBOX + off + 8 * h);
                    const float v[4] = {__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u),
                                        __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u)};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const f32x2 v2 = f2_make(v[e], v[e]);
#pragma unroll
                        for (int k = 0; k < N / 2; ++k) acc[k][e] = f2_fma(hw[j][k], v2, acc[k][e]);
                    }
                }
                // out streams 2k, 2k+1 replace residual streams 2k, 2k+1 (this
                // thread is the only reader and writer of its row's chunk)
#pragma unroll
                for (int k = 0; k < N / 2; ++k) {
                    float o0[4], o1[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) f2_split(acc[k][e], o0[e], o1[e]);
                    const uint32_t pw[4] = {pack2(o0[0], o0[1]), pack2(o0[2], o0[3]),
                                            pack2(o1[0], o1[1]), pack2(o1[2], o1[3])};
                    asm volatile("st.shared.v2.u32 [%0], {%1,%2};" ::"r"(st + 2 * k * P::XBOX + off + 8 * h),
                                 "r"(pw[0]), "r"(pw[1])
                                 : "memory");
                    asm volatile("st.shared.v2.u32 [%0], {%1,%2};" ::"r"(st + (2 * k + 1) * P::XBOX + off + 8 * h),
                                 "r"(pw[2]), "r"(pw[3])
                                 : "memory");
                    // the sum of squares of the stored (bf16) values, channel pairs
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const f32x2 ov = f2_make(__uint_as_float(pw[e] << 16),
                                                 __uint_as_float(pw[e] & 0xffff0000u));
                        ssq2 = f2_fma(ov, ov, ssq2);
                    }
                }
            }
            tc::fence_proxy_async_smem();
            tc::mbar_release(&ready[s]);
            // end of a group: this warp's half of the out.W'_hi buffer added to
            // the fp32 sum in TMEM
            const int g = i / P::G, hb = g & 1;
            if (i % P::G == P::G - 1 || i == ncb - 1) {
                if (*abort_v ||
                    !tc::mbar_wait(&hifull[hb], (g >> 1) & 1, fault, tc::kFaultTimeoutAcc)) {
                    *abort_v = 1;
                    ok = false;
                    break;
                }
                tc::tc_fence_after();
                const uint32_t hcol = trow + (hb ? P::HI1 : P::HI0) + hf * OH;
#pragma unroll
                for (int c8 = 0; c8 < OH / 8; ++c8) {
                    float w[8], a[8];
                    if (g == 0) {
                        tc::tmem_ld8_wait(hcol + c8 * 8, w);
                    } else {
                        tc::tmem_ld8x2_wait(ucol + c8 * 8, hcol + c8 * 8, a, w);
#pragma unroll
                        for (int e = 0; e < 8; ++e) w[e] = a[e] + w[e];
                    }
                    tc::tmem_st8_wait(ucol + c8 * 8, w);
                }
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&hiempty[hb]);
            }
        }
        // the row's sum of squares: half 1 hands its part to half 0
        float ssq_lo, ssq_hi;
        f2_split(ssq2, ssq_lo, ssq_hi);
        const float ssq = ssq_lo + ssq_hi;
        if (hf == 1) ssq_red[r] = ssq;
        tc::named_bar_sync(1 + q, 64);
        const float ssq_row = ssq + ssq_red[r];
        if (ok && !tc::mbar_wait(&acc_bar, 0, fault, tc::kFaultTimeoutAcc)) ok = false;
        tc::tc_fence_after();
        // u = sum over groups of out.W'_hi + (out.W'_lo + out.W'_lo2), this warp's half
        const bool store = ok && !*abort_v && live;
        float4 *dst = reinterpret_cast<float4 *>(upart + (int64_t(split) * T + t) * O + hf * OH);
#pragma unroll
        for (int c8 = 0; c8 < OH / 8; ++c8) {
            float w[8], w2[8], a[8];
            const uint32_t col = trow + P::LO + hf * OH + c8 * 8;
            tc::tmem_ld8x2_wait(col, col + O, w, w2);
            tc::tmem_ld8_wait(ucol + c8 * 8, a);
#pragma unroll
            for (int e = 0; e < 8; ++e) a[e] += w[e] + w2[e];
            if (store) {
                dst[2 * c8] = make_float4(a[0], a[1], a[2], a[3]);
                dst[2 * c8 + 1] = make_float4(a[4], a[5], a[6], a[7]);
            }
        }
        if (store && hf == 0) spart[int64_t(split) * T + t] = ssq_row;
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) tc::tmem_dealloc(tmem, P::TMEM_COLS);
}

// W [n C][O] fp32 -> for each BC-channel block, the shared-memory image of
// the fused kernel's W stage, so that one bulk copy loads it: for stream j,
// rows r = part O + o (the hi, lo, lo2 terms of W[j C + c][o]; zero rows
// past 3 O), BC channels per row in the stage's swizzle (P::chunk_off, for
// boxes aligned to the swizzle atom); channels past C are zero.  Block
// (cb, j): the BC x O source floats are one coalesced read into shared memory
// (rows padded against bank conflicts).
template <class P>
__global__ void __launch_bounds__(256) k_w_tile(const float *__restrict__ W, bf16 *__restrict__ Wt,
                                                int64_t C)
{
    pdl_wait();
    constexpr int O = P::O, OP = O + 1, CHUNKS = P::BC / 8;
    __shared__ float ws[P::BC * OP];
    const int cb = int(blockIdx.x), j = int(blockIdx.y);
    const int64_t c0 = int64_t(cb) * P::BC;
    const int cn = int(C - c0 < P::BC ? C - c0 : P::BC);
    const float *src = W + (int64_t(j) * C + c0) * O;
    for (int i = threadIdx.x; i < P::BC * O; i += blockDim.x) {
        const int c = i / O, o = i % O;
        ws[c * OP + o] = c < cn ? __ldg(src + i) : 0.f;
    }
    __syncthreads();
    uint8_t *dst = reinterpret_cast<uint8_t *>(Wt) + (int64_t(cb) * P::N + j) * P::WBOX;
    // item: output o and 16-byte chunk cc; its three terms go to rows o,
    // O + o and 2O + o (zero rows past 3O by the items that follow)
    for (int it = threadIdx.x; it < CHUNKS * O; it += blockDim.x) {
        const int cc = it / O, o = it % O;
        float hi[8], lo[8], lo2[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) w_terms(ws[(8 * cc + e) * OP + o], hi[e], lo[e], lo2[e]);
        *reinterpret_cast<uint4 *>(dst + P::chunk_off(o, cc)) = pack8(hi);
        *reinterpret_cast<uint4 *>(dst + P::chunk_off(O + o, cc)) = pack8(lo);
        *reinterpret_cast<uint4 *>(dst + P::chunk_off(2 * O + o, cc)) = pack8(lo2);
    }
    if constexpr (P::NB > 3 * O) {
        constexpr int ZR = P::NB - 3 * O;
        for (int it = threadIdx.x; it < CHUNKS * ZR; it += blockDim.x) {
            const int cc = it / ZR, r = 3 * O + it % ZR;
            *reinterpret_cast<uint4 *>(dst + P::chunk_off(r, cc)) = make_uint4(0, 0, 0, 0);
        }
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
// bf16 tensor of `rank` dims (innermost first) in the stage's swizzle
static bool map_bf16(CUtensorMap *m, const void *base, int rank, const uint64_t *dims,
                     const uint64_t *strides_bytes, const uint32_t *box, CUtensorMapSwizzle sw)
{
    return tmap_bf16(m, base, rank, dims, strides_bytes, box, sw);
}

// Channel-block splits: about one CTA per SM (the CTA fills most of shared
// memory); in batch-invariant mode fixed 1024-channel splits, so a
// token's sums do not depend on T.
static int post_proj_splits(int64_t T, int n, int64_t C)
{
    const int bc = n == 4 ? PostProj::BC : PostProj8::BC, minb = n == 4 ? PostProj::MINB : 1;
    const int64_t mt = (T + 127) / 128, cb = (C + bc - 1) / bc;
    int64_t s = batch_invariant() ? (cb * bc + 1023) / 1024
                                  : int64_t(kSplitSms) * minb / (mt > 0 ? mt : 1);
    if (s < 1) s = 1;
    if (s > cb) s = cb;
    return int(s);
}

// the split W: the tiled stage images
static size_t post_proj_w_bytes(int n, int64_t C)
{
    if (n == 8) return size_t((C + PostProj8::BC - 1) / PostProj8::BC) * PostProj8::WSTAGE;
    return size_t((C + PostProj::BC - 1) / PostProj::BC) * PostProj::N * PostProj::WBOX;
}

template <class P>
static cudaError_t launch_w_tile(const float *Wn, bf16 *Wt, int64_t C, cudaStream_t s)
{
    MHC_PROF("k_w_tile", s);
    launch_k(k_w_tile<P>, dim3(unsigned((C + P::BC - 1) / P::BC), unsigned(P::N)), dim3(256), 0, s,
             Wn, Wt, C);
    return cudaGetLastError();
}

// workspace: the split W, partials upart [S][T][O], spart [S][T]
size_t post_proj_ws_bytes(int64_t T, int n, int64_t C)
{
    const int64_t O = int64_t(n) * n + 2 * n;
    const int64_t S = post_proj_splits(T, n, C);
    return ws_align(post_proj_w_bytes(n, C)) + ws_align(size_t(S * T * O) * 4) +
           ws_align(size_t(S * T) * 4);
}

// n = 4: W tiled into stage images, then maps for x, f and out (BC-channel
// boxes in the stage's swizzle)
static cudaError_t post_proj4_launch(const bf16 *res, const bf16 *f, const bf16 *bias,
                                     const float *Hres, const float *Hpost, const float *Wn,
                                     bf16 *Wt, bf16 *out, float *upart, float *spart, int64_t T,
                                     int64_t C, int S, int *S_used_out, int *fault, cudaStream_t s)
{
    using P = PostProj;
    constexpr int n = P::N;
    const CUtensorMapSwizzle sw = P::BC == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    const uint64_t uC = uint64_t(C), uT = uint64_t(T);
    cudaError_t e = launch_w_tile<P>(Wn, Wt, C, s);
    if (e != cudaSuccess) return e;
    CUtensorMap tmx, tmf, tmo;
    {
        const uint64_t dims[3] = {uC, uint64_t(n), uT};
        const uint64_t strides[2] = {uC * 2, uC * 2 * n};
        const uint32_t box[3] = {P::BC, 1, P::BM};
        if (!map_bf16(&tmx, res, 3, dims, strides, box, sw) ||
            !map_bf16(&tmo, out, 3, dims, strides, box, sw))
            return cudaErrorInvalidValue;
    }
    {
        const uint64_t dims[2] = {uC, uT};
        const uint64_t strides[1] = {uC * 2};
        const uint32_t box[2] = {P::BC, P::BM};
        if (!map_bf16(&tmf, f, 2, dims, strides, box, sw)) return cudaErrorInvalidValue;
    }
    e = set_smem_limit(reinterpret_cast<const void *>(k_post_proj_tc<P>), P::SMEM);
    if (e != cudaSuccess) return e;
    const int cb_total = int((C + P::BC - 1) / P::BC);
    const int cps = (cb_total + S - 1) / S;
    *S_used_out = (cb_total + cps - 1) / cps;
    MHC_PROF("k_post_proj_tc", s);
    launch_k(k_post_proj_tc<P>, dim3(unsigned((T + P::BM - 1) / P::BM), unsigned(*S_used_out)),
             dim3(P::THREADS), P::SMEM, s, tmx, tmf, tmo, static_cast<const bf16 *>(Wt), bias, Hres,
             Hpost, upart, spart, T, C, cps, cb_total, fault);
    return cudaGetLastError();
}

// n = 8: W tiled into stage images, then maps for x and out (16-channel
// boxes, 32-byte swizzle) and bias ([1][C], boxes of 16)
static cudaError_t post_proj8_launch(const bf16 *res, const bf16 *f, const bf16 *bias,
                                     const float *Hres, const float *Hpost, const float *Wn,
                                     bf16 *Wt, bf16 *out, float *upart, float *spart, int64_t T,
                                     int64_t C, int S, int *S_used_out, int *fault, cudaStream_t s)
{
    using P = PostProj8;
    constexpr int n = P::N;
    const uint64_t uC = uint64_t(C), uT = uint64_t(T);
    const int cb_total = int((C + P::BC - 1) / P::BC);
    cudaError_t e = launch_w_tile<P>(Wn, Wt, C, s);
    if (e != cudaSuccess) return e;
    CUtensorMap tmx, tmb, tmo;
    {
        const uint64_t dims[3] = {uC, uint64_t(n), uT};
        const uint64_t strides[2] = {uC * 2, uC * 2 * n};
        const uint32_t box[3] = {P::BC, 1, P::BM};
        if (!map_bf16(&tmx, res, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_32B) ||
            !map_bf16(&tmo, out, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_32B))
            return cudaErrorInvalidValue;
    }
    std::memset(&tmb, 0, sizeof tmb);
    if (bias && !tmap_bf16_2d(&tmb, bias, 1, uC, 1, P::BC, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    CUtensorMap tmxp, tmfp;   // L2 prefetch boxes of PF_C channels
    {
        const uint64_t dims[3] = {uC, uint64_t(n), uT};
        const uint64_t strides[2] = {uC * 2, uC * 2 * n};
        const uint32_t box[3] = {P::PF_C, 1, P::BM};
        if (!map_bf16(&tmxp, res, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE) ||
            !tmap_bf16_2d(&tmfp, f, uT, uC, P::BM, P::PF_C, CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    }
    e = set_smem_limit(reinterpret_cast<const void *>(k_post_proj8_tc), P::SMEM);
    if (e != cudaSuccess) return e;
    const int cps = (cb_total + S - 1) / S;
    *S_used_out = (cb_total + cps - 1) / cps;
    MHC_PROF("k_post_proj8_tc", s);
    launch_k(k_post_proj8_tc, dim3(unsigned((T + P::BM - 1) / P::BM), unsigned(*S_used_out)),
             dim3(P::THREADS), P::SMEM, s, tmx, tmb, tmo, tmxp, tmfp, static_cast<const bf16 *>(Wt), f, bias,
             Hres, Hpost, upart, spart, T, C, cps, cb_total, fault);
    return cudaGetLastError();
}

cudaError_t launch_post_proj_fwd(const bf16 *res, const bf16 *f, const bf16 *bias,
                                 const float *Hres, const float *Hpost, const float *Wn,
                                 const float *alphan, const float *bn, int64_t T, int n,
                                 int64_t C, int iters, float eps_sk, float eps_rms, bf16 *out,
                                 float *Hpre_n, float *Hpost_n, float *Hres_n, float *u_save_n,
                                 float *r_save_n, void *ws, int *fault, cudaStream_t s)
{
    const int64_t O = int64_t(n) * n + 2 * n;
    const int S = post_proj_splits(T, n, C);
    char *p = static_cast<char *>(ws);
    bf16 *Wsplit = reinterpret_cast<bf16 *>(p);
    p += ws_align(post_proj_w_bytes(n, C));
    float *upart = reinterpret_cast<float *>(p);
    p += ws_align(size_t(int64_t(S) * T * O) * 4);
    float *spart = reinterpret_cast<float *>(p);
    int S_used = 1;
    cudaError_t e;
    if (n == 4) {
        e = post_proj4_launch(res, f, bias, Hres, Hpost, Wn, Wsplit, out, upart, spart, T, C, S,
                              &S_used, fault, s);
    } else {
        e = post_proj8_launch(res, f, bias, Hres, Hpost, Wn, Wsplit, out, upart, spart, T, C, S,
                              &S_used, fault, s);
    }
    if (e != cudaSuccess) return e;
    return launch_compute_h_parts(upart, spart, S_used, alphan, bn, T, n, C, iters, eps_sk,
                                  eps_rms, Hpre_n, Hpost_n, Hres_n, u_save_n, r_save_n, s);
}

}  // namespace mhc

