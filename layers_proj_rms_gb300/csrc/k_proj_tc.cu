// Forward projection of proj_rms_compute_h on the 5th-generation tensor
// cores (tcgen05): per token t and K split s,
//   upart[s][t][o] = sum_{k in s} x[t][k] W[k][o],   spart[s][t] = sum_{k in s} x[t][k]^2.
//
// Megatron's fused projection runs this on TF32 MMA with split-K (RL-Kernel
// PR #383, follow-up commit on the Megatron mHC source).  Here the operands
// are bf16: x is already bf16, and W (fp32, 24 significant bits) is split
// into three bf16 terms W_hi = bf16(W), W_lo = bf16(W - W_hi), W_lo2 =
// bf16(W - W_hi - W_lo), stacked as 3*O rows (zero-padded to a multiple of
// 16) of one B operand.  One MMA gives x.W_hi, x.W_lo and x.W_lo2; every
// product of bf16 values is exact in the fp32 accumulator and the three
// terms carry W to ~2^-24 relative.  (Two terms leave ~2^-17 of W per
// product, which at alpha = 1 and K = 57344 moves H by ~3e-5.)
//
// What remains is the accumulation.  The tensor core's fp32 accumulator
// loses about an ulp of the running sum per K step (measured on GB300: u's
// error grows with the number of K steps a split accumulates, ~1e-4 after
// 112 steps at |u| ~ 50), so the large x.W_hi term is never accumulated
// across k-blocks in TMEM: each 64-wide k-block's x.W_hi goes to one of two
// TMEM buffers and the epilogue warps add it into fp32 registers (round to
// nearest) while the MMAs fill the other buffer.  x.W_lo and x.W_lo2 (2^-8
// and 2^-16 of the sum) accumulate over the whole split in a third
// accumulator, whose accumulation error is that much smaller.
//
// CTA: BM tokens (128 at n = 4, 256 at n = 8) x one K split (K splits chosen
// for about MINB CTAs per SM); 2 + BM/32 warps:
//   warp 0      TMA producer: x tile [BM x 64] and W_hl tile [NB x 64] per
//               stage, both in the 128-byte swizzle layout
//   warp 1      TMEM allocation, MMA issue (one thread; per k step and
//               128-row half: x.W_hi, x.W_lo, x.W_lo2 as three MMAs of N = NH
//               sharing the stage's W_hl operand), commits
//   warps 2..   per k-block: the sum of squares of their token rows from the
//               same smem tiles, then the k-block's x.W_hi from TMEM into
//               registers; finally the epilogue (TMEM -> partials)
// Every wait is bounded; a timeout reports a fault code and the CTA unwinds.
#include <atomic>

#include "launch.h"
#include "tc.cuh"
#include "tmap.h"

namespace mhc {

// A stage holds KBS consecutive 64-wide k-blocks (KBS boxes issued back to
// back, so each token row is read in KBS*128 contiguous bytes); STG stages;
// MINB CTAs per SM; BM tokens per CTA, in MMAs of 128 rows that share the
// stage's W_hl tile (BM = 256 at n = 8, where the W_hl tile of a k-block,
// 240 rows, is larger than 128 rows of x).
template <int N, int KBS_, int STG_, int MINB_, int BM_ = 128, int G_ = 1>
struct ProjTcCfg {
    static constexpr int G = G_;   // stages per x.W_hi buffer (drained every G stages)
    static constexpr int O = N * N + 2 * N;
    static constexpr int NB = w_split_rows(N);  // MMA N: hi, lo, lo2 rows, zero rows (80 or 240)
    static constexpr int BM = BM_, BK = 64, KBS = KBS_, STAGES = STG_, MINB = MINB_;
    static constexpr int MH = BM / 128;               // MMAs of 128 rows per k step
    static constexpr int A_SUB = BM * BK * 2;
    static constexpr int B_SUB = NB * BK * 2;
    static constexpr int A_BYTES = KBS * A_SUB;
    static constexpr int STAGE = KBS * (A_SUB + B_SUB);  // multiple of 1024
    // TMEM per 128-row half: HB x.W_hi buffers of NH columns (NH = O
    // rounded up to 16: 32 / 80) and the accumulator of [x.W_lo | x.W_lo2]
    // (NL = 2O columns: W_hl rows [O, 3O) in one MMA).  n = 4: two x.W_hi
    // buffers; n = 8 (two halves of 240 columns in 512): one.
    static constexpr int NH = (O + 15) / 16 * 16, NL = 2 * O;
    static constexpr int HB = 3 * NH + NL <= 256 / MH ? 2 : 1;
    static constexpr int HI0 = 0, HI1 = NH, LO = HB * NH;
    static constexpr int ACC_COLS = LO + NL <= 128 ? 128 : 256;   // TMEM columns per half
    static constexpr int TMEM_COLS = MH * ACC_COLS;
    static_assert(LO + NL <= ACC_COLS && NH <= NB && 3 * O <= NB && NL % 16 == 0, "accumulators");
    static constexpr int EPI_WARPS = 4 * MH;
    static constexpr int THREADS = 64 + 32 * EPI_WARPS;
    static constexpr int SMEM = STAGES * STAGE + 1024 /*align*/ + 512 /*barriers*/;
    static_assert(A_SUB % 1024 == 0 && B_SUB % 1024 == 0, "sub-tiles keep 1024-byte alignment");
    static_assert(BM == 128 || BM == 256, "tile rows");
    static_assert(SMEM * MINB <= 232448, "shared memory");
};
template <int N> struct ProjTcSel;
// x.W_hi drained every 4 stages (16 K steps): at n = 8 draining every stage
// took 0.244 ms for the op at T=8192, C=7168, every 4 stages 0.232, every 8
// 0.230, with the error on u growing from 1.0e-5 to 2.3e-5 (alpha = 1,
// K = 57344); three separate MMAs of N = 80 for hi, lo and lo2 (x read from
// shared memory three times) took 0.29.
template <> struct ProjTcSel<4> { using type = ProjTcCfg<4, 1, 4, 2, 128, 4>; };
template <> struct ProjTcSel<8> { using type = ProjTcCfg<8, 1, 3, 1, 256, 4>; };
template <int N>
using ProjTc = typename ProjTcSel<N>::type;

// W [K][O] fp32 -> W_hl [NB][K] bf16 (rows o: hi; rows O+o: lo; rows 2O+o:
// lo2; rows 3O..NB: zero).  n = 4: one thread per k (the tiled form below,
// with 256 blocks, was slower at n = 4).
__global__ void k_w_split4(const float *__restrict__ W, bf16 *__restrict__ Whl, int64_t K)
{
    pdl_wait();
    constexpr int O = 24, NB = w_split_rows(4);
    const int64_t k = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (k >= K) return;
#pragma unroll 4
    for (int o = 0; o < O; ++o) {
        float hi, lo, lo2;
        w_terms(__ldg(W + k * O + o), hi, lo, lo2);
        Whl[int64_t(o) * K + k] = __float2bfloat16_rn(hi);
        Whl[int64_t(O + o) * K + k] = __float2bfloat16_rn(lo);
        Whl[int64_t(2 * O + o) * K + k] = __float2bfloat16_rn(lo2);
    }
#pragma unroll
    for (int o = 3 * O; o < NB; ++o) Whl[int64_t(o) * K + k] = __float2bfloat16_rn(0.f);
}

// n = 8: a block transposes a tile of 64 k rows through shared memory:
// the tile's 64*O floats are one contiguous, coalesced read, and each thread
// writes 8 consecutive k of one output row (16 bytes); the tile's rows are
// padded to O + 1 floats against bank conflicts.  Reading W[k][o] with one
// thread per k (a 4*O-byte stride across the lanes) took 23 us at n = 8.
constexpr int kWsplitK = 64;
template <int N>
__global__ void __launch_bounds__(256) k_w_split(const float *__restrict__ W, bf16 *__restrict__ Whl,
                                                 int64_t K)
{
    pdl_wait();
    constexpr int O = N * N + 2 * N;
    constexpr int OP = O + 1;   // padded row: the 8 lanes of one output row, 8 rows apart, use 4 banks
    __shared__ float ws[kWsplitK * OP];
    const int64_t k0 = int64_t(blockIdx.x) * kWsplitK;
    const int kn = int(K - k0 < kWsplitK ? K - k0 : kWsplitK);   // a multiple of 8
    for (int i = threadIdx.x; i < kn * O; i += blockDim.x) ws[(i / O) * OP + i % O] = __ldg(W + k0 * O + i);
    __syncthreads();
    // item: output o and 8-wide group kg of the tile's k; its three terms go
    // to rows o, O + o and 2O + o (zero rows past 3O, if any, by the items
    // that follow)
    constexpr int NB = w_split_rows(N);
    constexpr int KG = kWsplitK / 8;
    for (int it = threadIdx.x; it < O * KG; it += blockDim.x) {
        const int o = it / KG, kg = it % KG;
        if (kg * 8 >= kn) continue;
        float hi[8], lo[8], lo2[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) w_terms(ws[(kg * 8 + e) * OP + o], hi[e], lo[e], lo2[e]);
        bf16 *dst = Whl + int64_t(o) * K + k0 + kg * 8;
        *reinterpret_cast<uint4 *>(dst) = pack8(hi);
        *reinterpret_cast<uint4 *>(dst + int64_t(O) * K) = pack8(lo);
        *reinterpret_cast<uint4 *>(dst + int64_t(2 * O) * K) = pack8(lo2);
    }
    for (int it = threadIdx.x; it < (NB - 3 * O) * KG; it += blockDim.x) {
        const int ro = 3 * O + it / KG, kg = it % KG;
        if (kg * 8 >= kn) continue;
        *reinterpret_cast<uint4 *>(Whl + int64_t(ro) * K + k0 + kg * 8) = make_uint4(0, 0, 0, 0);
    }
}

template <int N, class P>
__global__ void __launch_bounds__(P::THREADS, P::MINB)
    k_proj_tc(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmw,
              float *__restrict__ upart, float *__restrict__ spart, int64_t T, int kb_per_split,
              int kb_total, int *fault)
{
    pdl_wait();
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + P::STAGES * P::STAGE);
    uint64_t *empty = full + P::STAGES;
    uint64_t *acc_bar = empty + P::STAGES;
    uint64_t *hifull = acc_bar + 1;     // [HB] a group's x.W_hi is in buffer b
    uint64_t *hiempty = hifull + 2;     // [HB] the epilogue has drained buffer b
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(hiempty + 2);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t m0 = int64_t(blockIdx.x) * P::BM;
    const int split = blockIdx.y;
    const int kb0 = split * kb_per_split;  // kb_per_split is a multiple of KBS
    const int kb1 = min(kb_total, kb0 + kb_per_split);
    const int nkb = (kb1 - kb0 + P::KBS - 1) / P::KBS;  // stages; a partial last one reads zeros

    if (threadIdx.x == 0) {
        for (int s = 0; s < P::STAGES; ++s) {
            tc::mbar_init(&full[s], 1);
            // the MMAs' commit + every epilogue thread once it has read the
            // stage (tc::mbar_release)
            tc::mbar_init(&empty[s], 1 + 32 * P::EPI_WARPS);
        }
        tc::mbar_init(acc_bar, 1);
        for (int hb = 0; hb < 2; ++hb) {
            tc::mbar_init(&hifull[hb], 1);
            tc::mbar_init(&hiempty[hb], P::EPI_WARPS);
        }
        *abort_flag = 0;
        tc::fence_barrier_init();
        tc::tma_prefetch_desc(&tmx);
        tc::tma_prefetch_desc(&tmw);
    }
    if (warp == 1) tc::tmem_alloc(tmem_slot, P::TMEM_COLS);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            int issued = 0;
            for (int i = 0; i < nkb && !*abort_flag; ++i) {
                const int s = i % P::STAGES;
                if (i >= P::STAGES &&
                    !tc::mbar_wait(&empty[s], ((i / P::STAGES) & 1) ^ 1, fault,
                                   tc::kFaultTimeoutEmpty)) {
                    *abort_flag = 1;
                    break;
                }
                uint8_t *st = smem + s * P::STAGE;
                tc::mbar_arrive_expect_tx(&full[s], P::STAGE);
                for (int j = 0; j < P::KBS; ++j)
                    tc::tma_load_2d(st + j * P::A_SUB, &tmx, (kb0 + i * P::KBS + j) * P::BK,
                                    int(m0), &full[s]);
                for (int j = 0; j < P::KBS; ++j)
                    tc::tma_load_2d(st + P::A_BYTES + j * P::B_SUB, &tmw,
                                    (kb0 + i * P::KBS + j) * P::BK, 0, &full[s]);
                issued = i + 1;
            }
            // do not leave while copies into this CTA's shared memory are in flight
            for (int i = max(0, issued - P::STAGES); i < issued; ++i)
                tc::mbar_wait(&full[i % P::STAGES], (i / P::STAGES) & 1, fault,
                              tc::kFaultTimeoutMisc);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc_hi = tc::idesc_bf16_f32(128, P::NH);
            constexpr uint32_t idesc_lo = tc::idesc_bf16_f32(128, P::NL);
            constexpr int O = P::O;
            for (int i = 0; i < nkb; ++i) {
                // stage i belongs to group g = i / G, whose x.W_hi goes to buffer hb
                const int s = i % P::STAGES, g = i / P::G, hb = g % P::HB;
                const bool first = i % P::G == 0, last = i % P::G == P::G - 1 || i == nkb - 1;
                if (*abort_flag ||
                    !tc::mbar_wait(&full[s], (i / P::STAGES) & 1, fault, tc::kFaultTimeoutFull)) {
                    *abort_flag = 1;
                    break;
                }
                tc::tc_fence_after();
                const uint32_t a0 = tc::smem_u32(smem + s * P::STAGE);
                // [x.W_lo | x.W_lo2] first (W_hl rows [O, 3O): a multiple of 8
                // rows, so the operand starts on a 1024-byte swizzle group),
                // which keeps the tensor cores busy while the epilogue drains
                // the x.W_hi buffer
#pragma unroll
                for (int j = 0; j < P::KBS; ++j) {
                    const uint32_t a = a0 + j * P::A_SUB, b = a0 + P::A_BYTES + j * P::B_SUB;
#pragma unroll
                    for (int kk = 0; kk < P::BK / 16; ++kk)
#pragma unroll
                        for (int h = 0; h < P::MH; ++h)
                            tc::mma_bf16(tmem + h * P::ACC_COLS + P::LO,
                                         tc::desc_kmajor_sw128(a + h * 128 * 128 + kk * 32),
                                         tc::desc_kmajor_sw128(b + O * 128 + kk * 32), idesc_lo,
                                         (i > 0 || j > 0 || kk > 0) ? 1u : 0u);
                }
                // x.W_hi buffer hb must have been drained (group g - HB)
                if (first && g >= P::HB &&
                    !tc::mbar_wait(&hiempty[hb], ((g / P::HB) - 1) & 1, fault,
                                   tc::kFaultTimeoutAcc)) {
                    *abort_flag = 1;
                    break;
                }
                tc::tc_fence_after();
#pragma unroll
                for (int j = 0; j < P::KBS; ++j) {
                    const uint32_t a = a0 + j * P::A_SUB, b = a0 + P::A_BYTES + j * P::B_SUB;
#pragma unroll
                    for (int kk = 0; kk < P::BK / 16; ++kk)
#pragma unroll
                        for (int h = 0; h < P::MH; ++h)
                            tc::mma_bf16(tmem + h * P::ACC_COLS + (hb ? P::HI1 : P::HI0),
                                         tc::desc_kmajor_sw128(a + h * 128 * 128 + kk * 32),
                                         tc::desc_kmajor_sw128(b + kk * 32), idesc_hi,
                                         (!first || j > 0 || kk > 0) ? 1u : 0u);
                }
                tc::mma_commit(&empty[s]);
                if (last) tc::mma_commit(&hifull[hb]);
            }
            tc::mma_commit(acc_bar);
            tc::mbar_wait(acc_bar, 0, fault, tc::kFaultTimeoutAcc);
        }
        __syncwarp();
    } else {
        // warps 2..: token row r of the tile; TMEM lane r % 128 of accumulator r / 128
        const int q = warp & 3;
        const int hh = (warp - 2) >> 2;
        const int r = hh * 128 + q * 32 + lane;
        const uint32_t trow = tmem + hh * P::ACC_COLS + (uint32_t(q * 32) << 16);
        constexpr int O = P::O;
        float ssq = 0.f;
        float uhi[O];   // sum over this split's k-blocks of x.W_hi, in fp32 (round to nearest)
#pragma unroll
        for (int o = 0; o < O; ++o) uhi[o] = 0.f;
        bool ok = true;
        for (int i = 0; i < nkb; ++i) {
            const int s = i % P::STAGES;
            if (*abort_flag ||
                !tc::mbar_wait(&full[s], (i / P::STAGES) & 1, fault, tc::kFaultTimeoutFull)) {
                *abort_flag = 1;
                ok = false;
                break;
            }
            // The row's eight 16-byte chunks, in an order that differs per
            // lane: rows that share banks (r and r+8, r+16, ...) then read
            // different chunks, so a warp's loads are free of bank conflicts.
            // The sum of squares does not depend on the order.
#pragma unroll
            for (int j = 0; j < P::KBS; ++j) {
                const uint32_t row = tc::smem_u32(smem + s * P::STAGE + j * P::A_SUB + r * 128);
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    float f[8];
                    unpack8(lds128(row + (c ^ (lane & 7)) * 16), f);
#pragma unroll
                    for (int e = 0; e < 8; ++e) ssq = fmaf(f[e], f[e], ssq);
                }
            }
            tc::mbar_release(&empty[s]);
            // at the end of a group: its x.W_hi into the registers, then the
            // buffer goes back
            const int g = i / P::G, hb = g % P::HB;
            if (i % P::G != P::G - 1 && i != nkb - 1) continue;
            if (*abort_flag ||
                !tc::mbar_wait(&hifull[hb], (g / P::HB) & 1, fault, tc::kFaultTimeoutAcc)) {
                *abort_flag = 1;
                ok = false;
                break;
            }
            tc::tc_fence_after();
#pragma unroll
            for (int c = 0; c < P::NH / 16; ++c) {
                float w[16];
                tc::tmem_ld16_wait(trow + (hb ? P::HI1 : P::HI0) + c * 16, w);
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    if (c * 16 + e < O) uhi[c * 16 + e] += w[e];
            }
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&hiempty[hb]);
        }
        if (ok && !tc::mbar_wait(acc_bar, 0, fault, tc::kFaultTimeoutAcc)) ok = false;
        tc::tc_fence_after();
        const int64_t t = m0 + r;
        // u = sum over groups of x.W_hi + (x.W_lo + x.W_lo2)
        {
            float lo[O];
#pragma unroll
            for (int c = 0; c < O / 8; ++c) {
                float w[8], w2[8];
                tc::tmem_ld8x2_wait(trow + P::LO + c * 8, trow + P::LO + O + c * 8, w, w2);
#pragma unroll
                for (int e = 0; e < 8; ++e) lo[c * 8 + e] = w[e] + w2[e];
            }
#pragma unroll
            for (int o = 0; o < O; ++o) uhi[o] += lo[o];
        }
        if (ok && t < T) {
            float4 *dst = reinterpret_cast<float4 *>(upart + (int64_t(split) * T + t) * O);
#pragma unroll
            for (int o4 = 0; o4 < O / 4; ++o4)
                dst[o4] = make_float4(uhi[4 * o4], uhi[4 * o4 + 1], uhi[4 * o4 + 2], uhi[4 * o4 + 3]);
            spart[int64_t(split) * T + t] = ssq;
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) tc::tmem_dealloc(tmem, P::TMEM_COLS);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
// Batch-invariant mode: the K splits depend on K alone (fixed 4096-wide
// splits), so a token's u and s, and everything computed from them, do not
// depend on how many tokens share the call.  Otherwise the split count is
// chosen for about MINB CTAs per SM, which depends on T.
// The flag is process-wide and atomic: a thread that sets it while another
// launches reads either value, never a torn one (calls that must see the new
// mode should be ordered after the setter by the caller).
static std::atomic<int> g_batch_invariant{0};

void set_batch_invariant(int on) { g_batch_invariant.store(on ? 1 : 0, std::memory_order_relaxed); }
int batch_invariant() { return g_batch_invariant.load(std::memory_order_relaxed); }

int proj_tc_splits(int64_t T, int n, int64_t K)
{
    const int bm = n == 4 ? ProjTc<4>::BM : ProjTc<8>::BM;
    const int64_t mt = (T + bm - 1) / bm;
    const int64_t kb = (K + 63) / 64;
    const int minb = n == 4 ? ProjTc<4>::MINB : ProjTc<8>::MINB;
    int64_t s = batch_invariant() ? (kb + 63) / 64
                                  : (int64_t(kSplitSms) * minb) / (mt > 0 ? mt : 1);
    if (s < 1) s = 1;
    if (s > kb) s = kb;
    if (s > 32) s = 32;
    return int(s);
}

// k-blocks per split, a multiple of the k-blocks per stage
static int proj_tc_kps(int64_t K, int S, int kbs)
{
    const int kb_total = int((K + 63) / 64);
    int kps = (kb_total + S - 1) / S;
    return (kps + kbs - 1) / kbs * kbs;
}

cudaError_t launch_w_split(const float *W, bf16 *Whl, int n, int64_t K, cudaStream_t s)
{
    MHC_PROF("k_w_split", s);
    if (n == 4)
        launch_k(k_w_split4, dim3(unsigned((K + 255) / 256)), dim3(256), 0, s, W, Whl, K);
    else
        launch_k(k_w_split<8>, dim3(unsigned((K + kWsplitK - 1) / kWsplitK)), dim3(256), 0, s, W,
                 Whl, K);
    return cudaGetLastError();
}

template <int N, class P>
static cudaError_t proj_tc_impl(const bf16 *x, const float *W, int64_t T, int64_t C, bf16 *Whl,
                                float *upart, float *spart, int S, int *fault, cudaStream_t s)
{
    const int64_t K = int64_t(N) * C;
    {
        cudaError_t e = launch_w_split(W, Whl, N, K, s);
        if (e != cudaSuccess) return e;
    }
    CUtensorMap tmx, tmw;
    if (!tmap_bf16_2d(&tmx, x, uint64_t(T), uint64_t(K), P::BM, P::BK,
                       CU_TENSOR_MAP_SWIZZLE_128B) ||
        !tmap_bf16_2d(&tmw, Whl, uint64_t(P::NB), uint64_t(K), P::NB, P::BK,
                       CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    cudaError_t e = set_smem_limit(reinterpret_cast<const void *>(k_proj_tc<N, P>), P::SMEM);
    if (e != cudaSuccess) return e;
    const int kb_total = int((K + P::BK - 1) / P::BK);
    const int kps = proj_tc_kps(K, S, P::KBS);
    const int S_used = (kb_total + kps - 1) / kps;
    dim3 grid(unsigned((T + P::BM - 1) / P::BM), unsigned(S_used));
    {
        MHC_PROF("k_proj_tc", s);
        launch_k(k_proj_tc<N, P>, dim3(grid), dim3(P::THREADS), P::SMEM, s, tmx, tmw, upart, spart,
                 T, kps, kb_total, fault);
    }
    return cudaGetLastError();
}

// Returns the number of K splits actually used (partials upart[0..S_used)).
cudaError_t launch_proj_partials(const bf16 *x, const float *W, int64_t T, int n, int64_t C,
                                 bf16 *Whl, float *upart, float *spart, int *splits_used,
                                 int *fault, cudaStream_t s)
{
    const int64_t K = int64_t(n) * C;
    const int S = proj_tc_splits(T, n, K);
    const int kb_total = int((K + 63) / 64);
    const int kps = proj_tc_kps(K, S, n == 4 ? ProjTc<4>::KBS : ProjTc<8>::KBS);
    *splits_used = (kb_total + kps - 1) / kps;
    if (n == 4) return proj_tc_impl<4, ProjTc<4>>(x, W, T, C, Whl, upart, spart, S, fault, s);
    return proj_tc_impl<8, ProjTc<8>>(x, W, T, C, Whl, upart, spart, S, fault, s);
}

}  // namespace mhc
