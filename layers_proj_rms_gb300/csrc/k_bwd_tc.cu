// Residual-gradient pass of the mHC layer backward on tcgen05 tensor cores.
//
// For a slice of CW channels across all n streams (a set of 128 flattened
// residual indices k = j*C + c) and a contiguous range of tokens, one CTA
// computes
//   dx[t][j][c] = sum_o du[t][o] W[k][o] + coef[t] x[t][j][c]
//               [+ H_pre[t][j] dy[t][c] + sum_i H_res[t][j][i] dout[t][i][c]]   (layer)
//   dW[k][o]   += sum_t x[t][k] du[t][o]
//   dbias[c]   += sum_t sum_i H_post[t][i] dout[t][i][c]                        (layer)
// i.e. the projection backward of RL-Kernel PR #383 (fp32_gemm_rms: dx_gemm
// + dx_rms, dW) fused with the aggregate and post-mix residual gradients and
// the three-way sum (Megatron-Core fused_mhc_kernels fused_add_3).
//
// du (fp32) arrives as bf16 hi | lo halves (du_hl[t][0..O) = bf16(du),
// du_hl[t][O..2O) = bf16(du - hi)), which together carry du to ~2^-17; W is
// split the same way into W_hi and W_lo.  The product below then differs from
// du.W^T by at most kSplitBound * sum_o |du_o| * max_ko |W_ko| (the dropped
// du_lo.W_lo, the remainders of du and W, the fp32 accumulation).  A token
// for which that bound exceeds kExactAbove (rows of near-zero RMS, where
// r = 1/(q + eps) makes du ~1e5 while dx stays O(1) through cancellation)
// takes the exact path instead: its du.W^T is recomputed in fp64 from the
// fp32 du and W, so dx meets the bf16 gradient tolerance on every token.
// Per tile of 128 tokens (MMA 1 first, so the epilogue's accumulator is
// complete before the dW and dbias MMAs of the tile run):
//   MMA 1 (dx_gemm): D2[t][k] = du_hi.W_hi + du_lo.W_hi + du_hi.W_lo (the
//          dropped du_lo.W_lo is ~2^-18 relative): M = 128 tokens, N = 128 k,
//          K = 2*O against Wd = [W_hi | W_hi], then K = O against W_lo
//          (n = 8: the du_lo steps reuse the W_hi steps' operand)
//   MMA 2 (dW):      D1[k][o'] += sum_t x[t][k] du_hl[t][o'], M = 128 k,
//          N = 2*O (n = 8: 128 + 32, one MMA per du_hl swizzle box),
//          K = tokens; hi and lo columns of D1 are summed at the end.
//          Both operands are read MN-major straight from the TMA tiles.
//   MMA 3 (n = 4, dbias): D3[k][o'] += sum_t dout[t][k] du_hl[t][o'] with
//          H_post hi | lo stored in du_hl columns [2O, 2O+2n)
//   epilogue: D2 + the elementwise terms -> dx (bf16), written over the x
//          chunk each thread has just read in the stage (the stage's stream
//          boxes have dx's layout), then stored by TMA.
// D2 is double-buffered in TMEM so the next tile's MMAs overlap the
// epilogue; D1 accumulates over the whole token range and is written as this
// split's dW partial.  Every input of a tile arrives by TMA ahead of its use:
// n = 4, x, dout, dy and du_hl in a ring of two stages (every DRAM access a
// whole 64-byte row), the per-token inputs copied by the epilogue with
// cp.async one tile ahead; n = 8 (16-channel slices, a 40 KB W tile), x in a
// ring of two stages and single buffers refilled a tile ahead: du_hl
// (released by the MMAs), the per-token inputs H_res, H_pre, H_post and dout
// and dy (released once the epilogue has read them).  Per-lane global loads
// of these inputs (each warp load touching 32 token rows) cost 2.8x the
// time at n = 8, and per-lane 16-byte dx stores half of the tile period.
// Warps: 0 the stage producer (n = 8: also the dx stores of a tile, right
// before it refills that stage), 1 TMEM + MMA issue, 2 (n = 8) the
// single-buffer producer, then the epilogue: CW/8 warps per TMEM lane
// quadrant, each thread one token row x one 8-channel chunk of every stream
// (16 epilogue warps for n = 4, 8 for n = 8; at n = 4 lanes of each
// quadrant's first warp store the quadrant's dx rows).  Before their first
// tile the epilogue warps build the slice's W tile in shared memory from
// fp32 W (bf16 hi/lo split, swizzled for the MMA).  An unsplit pass writes
// dW and dbias directly.
#include "launch.h"
#include "tc.cuh"
#include "tmap.h"

namespace mhc {

// Error bound factor of the two-term bf16 product (see above): the three
// dropped terms are each at most 2^-16 |du_o W_ko|, the fp32 accumulation
// over at most 16 K steps 2^-20.
constexpr float kSplitBound = 3.25f / 65536.f;
// Above this bound on |dx_gemm error| (a fifth of the 2e-2 absolute
// tolerance of the bf16 gradients) a token takes the exact path.
constexpr float kExactAbove = 4e-3f;

// The exact path's dot product of a token's fp32 du row with a row of W, in
// fp64: each product of two fp32 values is exact in fp64 and the O terms
// accumulate with ~2^-53 relative rounding.
__device__ __forceinline__ float exact_du_w(const float *__restrict__ du,
                                           const float *__restrict__ w, int O)
{
    double acc = 0.0;
#pragma unroll 1
    for (int o = 0; o < O; o += 4) {
        const float4 a = __ldg(reinterpret_cast<const float4 *>(du + o));
        const float4 b = __ldg(reinterpret_cast<const float4 *>(w + o));
        acc = fma(double(a.x), double(b.x), acc);
        acc = fma(double(a.y), double(b.y), acc);
        acc = fma(double(a.z), double(b.z), acc);
        acc = fma(double(a.w), double(b.w), acc);
    }
    return float(acc);
}

template <int N>
struct BwdTc {
    static constexpr int O = N * N + 2 * N;     // 24 / 80
    static constexpr int CW = 128 / N;          // channels per stream: 32 / 16
    static constexpr int CHUNKS = CW / 8;       // 8-channel chunks per stream slice: 4 / 2
    static constexpr int EPI_WARPS = 4 * CHUNKS;        // 16 / 8
    static constexpr int TT = 128;              // tokens per tile
    static constexpr int XROW = CW * 2;         // bytes of one token row of a stream box
    static constexpr uint32_t XSWZ = N == 4 ? tc::kSwz64 : tc::kSwz32;
    static constexpr int XBOX = TT * XROW;      // bytes of one stream box
    static constexpr int X_BYTES = N * XBOX;    // 32 KB
    // n = 4: one ring of stages holds x, dout, dy and du_hl of a tile.
    // n = 8: the ring holds x only; du_hl has one buffer that the MMAs release
    // as soon as they complete, and dout and dy one buffer (G) that the
    // epilogue releases once it has read them: both are refilled a tile ahead
    // in the shared memory that a second du_hl stage would take.
    static constexpr bool STAGE_G = N == 4;     // dout and dy in the ring
    static constexpr int G_BYTES = STAGE_G ? N * XBOX : 0;
    static constexpr int Y_BYTES = STAGE_G ? XBOX : 0;
    // du_hl tile: n = 4, one 128-byte-swizzled atom of 64 columns (hi [0,24) |
    // lo [24,48) | H_post hi, lo | zeros); n = 8, two such atoms (hi [0,80) |
    // lo [80,128)) and a 64-byte-swizzled tail box of columns [128,160)
    static constexpr int DU_ATOMS = N == 4 ? 1 : 2;
    static constexpr int DU_COLS = N == 4 ? 64 : 192;   // columns of du_hl in memory
    static constexpr int DU_ATOM_BYTES = TT * 128;
    static constexpr int DU_TAIL = DU_ATOMS * DU_ATOM_BYTES;
    static constexpr int DU_TAIL_BYTES = N == 4 ? 0 : TT * 64;
    static constexpr int DU_BYTES = DU_TAIL + DU_TAIL_BYTES;   // 16 KB / 40 KB
    static constexpr int G_OFF = X_BYTES, Y_OFF = G_OFF + G_BYTES, DU_OFF = Y_OFF + Y_BYTES;
    static constexpr int STAGE = N == 4 ? DU_OFF + DU_BYTES : X_BYTES;   // 88 KB / 32 KB
    static constexpr int STAGES = 2;
    // B operand of the dx GEMM.  n = 4: Wd = [W_hi | W_hi | W_lo | 0] in bf16,
    // planes of 64 columns (128-byte rows, 128-byte swizzle).  n = 8: a W_hi
    // plane (columns [0,64)), a W_lo plane, and a 64-byte-swizzled tail of
    // [W_hi [64,80) | W_lo [64,80)]; du_lo steps reuse the W_hi steps.
    static constexpr int NW = 2 * O;                    // 48 / 160
    static constexpr int KSTEP_A = NW / 16;             // du_hl . [W_hi | W_hi]: 3 / 10
    static constexpr int KSTEP_B = (O + 15) / 16;       // du_hi . W_lo: 2 / 5
    static constexpr int W_COLS = NW + 16 * KSTEP_B;    // 80 (n = 4)
    static constexpr int W_PLANES = N == 4 ? (W_COLS + 63) / 64 : 2;
    static constexpr int W_PLANE_BYTES = 128 * 128;
    static constexpr int W_TAIL = W_PLANES * W_PLANE_BYTES;
    static constexpr int W_BYTES = W_TAIL + (N == 4 ? 0 : 128 * 64);   // 32 KB / 40 KB
    static constexpr int DU1_OFF = STAGES * STAGE;      // n = 8: the du_hl buffer
    static constexpr int DU1_BYTES = N == 4 ? 0 : DU_BYTES;
    static constexpr int W_OFF = DU1_OFF + DU1_BYTES;
    static constexpr int D2_COL = 0, D1_COL = 256;      // D2 buffers at 0 and 128
    // n = 4: dbias on the tensor cores, D3[k][o'] += sum_t dout[t][k] du_hl[t][o'];
    // columns 2O+i (hi) and 2O+N+i (lo) of du_hl hold H_post[t][i]
    static constexpr int D3_COL = 320, D3_N = 64;
    static constexpr int TMEM_COLS = 512;
    // Per-token inputs of a tile in shared memory, one tile ahead.  n = 4:
    // the epilogue copies them with cp.async (H_res row, H_pre row: 20 floats
    // per token; coef).  n = 8 (layer): the producer loads them by TMA, H_res
    // transposed (the Hres argument is then HresT[t][i][j] = H_res[t][j][i],
    // which the compute_h backward writes, so that a dout stream's eight
    // weights are two 16-byte reads) as two 128-byte-swizzled boxes of 32
    // floats per token, H_pre and H_post as 32-byte-swizzled boxes of 8
    // floats (conflict-free row reads).
    static constexpr bool STAGE_P = N == 4;
    static constexpr bool TMA_P = N == 8;
    static constexpr int PAR_ROW = 20 * 4;
    static constexpr int PAR_OFF = W_OFF + W_BYTES;
    static constexpr int PH_PRE = 2 * TT * 128, PH_POST = PH_PRE + TT * 32;
    static constexpr int PAR_BYTES =
        STAGE_P ? TT * PAR_ROW + 2 * TT * 4 : (TMA_P ? PH_POST + TT * 32 : 0);   // 11 KB / 40 KB
    // n = 8 (layer): the G buffer, dout boxes of the n streams then the dy box
    static constexpr int G1_OFF = PAR_OFF + PAR_BYTES;
    static constexpr int G1_BYTES = N == 4 ? 0 : (N + 1) * XBOX;       // 36 KB
    static constexpr int SMEM = G1_OFF + G1_BYTES + 1024;
    // dx leaves through shared memory: the epilogue writes each dx chunk over
    // the x chunk it has just read (the stage's stream boxes have dx's
    // layout) and the rows go out by TMA store (whole rows, where per-lane
    // 16-byte global stores touched 32 token rows per warp instruction).
    // n = 8: the stage producer stores a tile's dx before it refills the
    // stage (the stores' reads of shared memory take a few thousand cycles,
    // which then stay off the epilogue).  n = 4: lanes of each TMEM lane
    // quadrant's first warp store the quadrant's rows (the 88 KB stage is
    // back sooner when the stores go out per quadrant).
    static constexpr bool STORER = N == 8;
    // Warps before the epilogue: 0 the stage producer (x ring; n = 8 also the
    // dx stores), 1 TMEM + MMA issue, 2 (n = 8) the single-buffer producer.
    static constexpr int NPRE = N == 8 ? 3 : 2;
    static constexpr int THREADS = 32 * NPRE + 32 * EPI_WARPS;  // 576 / 352
    // x is waited for where it is first read (the dW MMAs, the epilogue's
    // output phase), not before the dx GEMM and the mix, which do not read
    // it.  n = 4: the stage's x and its other part (dout, dy, du_hl: the G
    // part) have barriers of their own; the G part returns to the producer
    // once the epilogue's mix and the tile's MMAs are done with it, x once
    // the dx stores have read it.
    static constexpr bool SPLIT = N == 4;
    static_assert(STAGE % 1024 == 0 && DU_OFF % 1024 == 0 && PAR_OFF % 1024 == 0 &&
                      W_OFF % 1024 == 0 && (N == 4 || G1_OFF % 1024 == 0),
                  "alignment");
    static_assert(SMEM + 1024 <= 232448, "shared memory (dynamic + static)");
};

// Column sums over the 32 lanes of a warp: on entry every lane holds COLS
// values, on exit lane l holds the warp total of column (l % COLS).
template <int COLS>
__device__ __forceinline__ float warp_column_sum(float (&v)[COLS])
{
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int w = COLS / 2; w >= 1; w >>= 1) {
        const bool upper = (lane & w) != 0;
#pragma unroll
        for (int k = 0; k < w; ++k) {
            const float send = upper ? v[k] : v[k + w];
            const float keep = upper ? v[k + w] : v[k];
            v[k] = keep + __shfl_xor_sync(kFull, send, w);
        }
    }
    float r = v[0];
#pragma unroll
    for (int m = COLS; m < 32; m <<= 1) r += __shfl_xor_sync(kFull, r, m);
    return r;
}

struct BwdTcArgs {
    const float *W;    // [K][O] fp32
    const float *du32; // [T][O] fp32 du (the exact path)
    const float *dub;  // [T] sum_o |du[t][o]|
    const bf16 *dout, *dy;
    const float *coef, *Hpre, *Hres, *Hpost;
    bf16 *dx;
    float *dWpart;     // [splits][K][O]
    float *dbiaspart;  // [splits][C] (layer only)
    int64_t T, C;
    int tiles_per_split, tiles_total;
    int *fault;
};

// 16-byte chunk `chunk` of token row r of a stream box in the 64-byte (n=4)
// or 32-byte (n=8) swizzle layout that TMA writes.
template <int N>
__device__ __forceinline__ uint32_t box_chunk_addr(const uint8_t *box, int r, int chunk)
{
    constexpr int XROW = BwdTc<N>::XROW;
    const int phys = N == 4 ? (chunk ^ ((r >> 1) & 3)) : (chunk ^ ((r >> 2) & 1));
    return tc::smem_u32(box) + r * XROW + phys * 16;
}

template <int N>
__device__ __forceinline__ uint4 box_chunk(const uint8_t *box, int r, int chunk)
{
    return lds128(box_chunk_addr<N>(box, r, chunk));
}

template <int N, bool LAYER>
__global__ void __launch_bounds__(BwdTc<N>::THREADS, 1)
    k_bwd_tc(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmdu,
             const __grid_constant__ CUtensorMap tmg,
             const __grid_constant__ CUtensorMap tmy, const __grid_constant__ CUtensorMap tmdu2,
             const __grid_constant__ CUtensorMap tmhres, const __grid_constant__ CUtensorMap tmhpre,
             const __grid_constant__ CUtensorMap tmhpost, const __grid_constant__ CUtensorMap tmdx,
             const BwdTcArgs a)
{
    pdl_wait();
    using P = BwdTc<N>;
    constexpr int O = P::O, CW = P::CW;
    constexpr bool SG = LAYER && P::STAGE_G;
    constexpr bool TP = LAYER && P::TMA_P;    // per-token inputs by TMA (n = 8)
    constexpr bool G1 = LAYER && N == 8;      // dout and dy in the G buffer
    extern __shared__ uint8_t smem_raw[];
    // full: the stage has landed; empty: the tile's MMAs (n = 4: and the
    // epilogue warps, after the quadrants' dx stores have read it) are done
    // with it; xfree: the tile's dW MMAs have read its x; dxfull[s][0]
    // (n = 8): every epilogue thread has written its dx chunks into the stage
    // (and read what it needed); dxfull[s][q] (n = 4): quadrant q's threads
    __shared__ uint64_t full[P::STAGES], empty[P::STAGES], xfree[P::STAGES], dxfull[P::STAGES][4];
    // n = 4: the G part of a stage has landed / is free again
    __shared__ uint64_t gsfull[P::STAGES], gsempty[P::STAGES];
    __shared__ uint64_t wfull, d2full[2], d2empty[2], d1full, pfull, pempty, dufull, duempty,
        gfull, gempty;
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;
    __shared__ float bias_red[4][CW];
    __shared__ uint32_t wmax_bits;   // max |W| over the slice (bits of a nonnegative float)

    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *wtile = smem + P::W_OFF;
    volatile int *abort_v = &abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t C = a.C, K = int64_t(N) * C;
    const int64_t c0 = int64_t(blockIdx.x) * CW;
    const int split = blockIdx.y;
    const int tile0 = split * a.tiles_per_split;
    const int ntiles = min(a.tiles_total, tile0 + a.tiles_per_split) - tile0;
    // bytes of a stage's x part (n = 8: the whole stage) and of its G part (n = 4)
    constexpr uint32_t x_tx = P::X_BYTES;
    constexpr uint32_t g_tx = P::SPLIT ? (SG ? P::G_BYTES + P::Y_BYTES : 0) + P::DU_BYTES : 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < P::STAGES; ++s) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&empty[s], P::STORER ? 1 : 1 + P::EPI_WARPS);
            tc::mbar_init(&xfree[s], 1);
            // the MMAs' commit (+ one arrival per epilogue warp after the mix)
            tc::mbar_init(&gsfull[s], 1);
            tc::mbar_init(&gsempty[s], 1 + (LAYER ? P::EPI_WARPS : 0));
            // (the single buffers: every epilogue thread releases after its
            // own reads, tc::mbar_release)
            for (int q = 0; q < 4; ++q)
                tc::mbar_init(&dxfull[s][q], P::STORER ? 32 * P::EPI_WARPS : 32 * P::CHUNKS);
        }
        tc::mbar_init(&wfull, 32 * P::EPI_WARPS);
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(&d2full[b], 1);
            tc::mbar_init(&d2empty[b], P::EPI_WARPS);
        }
        tc::mbar_init(&d1full, 1);
        tc::mbar_init(&pfull, 1);
        tc::mbar_init(&pempty, 32 * P::EPI_WARPS);
        tc::mbar_init(&dufull, 1);
        tc::mbar_init(&duempty, 1);
        tc::mbar_init(&gfull, 1);
        tc::mbar_init(&gempty, 32 * P::EPI_WARPS);
        abort_flag = 0;
        wmax_bits = 0;
        tc::fence_barrier_init();
    }
    if (warp == 1) tc::tmem_alloc(&tmem_slot, P::TMEM_COLS);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------- stage producer
        // n = 8: before a stage is refilled, this warp stores the dx that the
        // epilogue wrote into it (lane j: stream j's box of the tile's 128
        // rows; rows past T and channels past C are clipped by the store)
        // and waits until the stores have read it.  Lane 0 waits and issues
        // the loads.
        if (lane == 0) {
            tc::tma_prefetch_desc(&tmx);
            tc::tma_prefetch_desc(&tmdx);
            if (N == 4) tc::tma_prefetch_desc(&tmdu);
            if (SG) {
                tc::tma_prefetch_desc(&tmg);
                tc::tma_prefetch_desc(&tmy);
            }
        }
        // lane 0 waits on `bar` (parity `par`); false (n = 8: for every lane)
        // after a failure
        auto lane0_wait = [&](uint64_t *bar, uint32_t par) -> bool {
            int go = 1;
            if (lane == 0) {
                go = !*abort_v && tc::mbar_wait(bar, par, a.fault, tc::kFaultTimeoutEmpty);
                if (!go) *abort_v = 1;
            }
            return P::STORER ? __shfl_sync(kFull, go, 0) != 0 : go != 0;
        };
        auto store_dx = [&](int k) -> bool {
            const int sk = k % P::STAGES;
            if (!lane0_wait(&dxfull[sk][0], (k / P::STAGES) & 1)) return false;
            if (lane < N) {
                tc::tma_store_3d(&tmdx, smem + sk * P::STAGE + lane * P::XBOX, int(c0), lane,
                                 (tile0 + k) * P::TT);
                tc::bulk_commit_group();
            }
            return true;
        };
        int issued = 0, stored = 0;   // x parts loaded; tiles whose dx was stored
        int gissued = 0;              // n = 4: G parts loaded
        bool good = true;
        // (n = 4: lane 0 alone)
        for (int i = 0; (P::STORER || lane == 0) && i < ntiles; ++i) {
            const int s = i % P::STAGES;
            if (P::SPLIT && lane == 0) {
                // n = 4: the G part first (the dx GEMM and the mix need it
                // before x)
                if (i >= P::STAGES) {
                    good = lane0_wait(&gsempty[s], ((i / P::STAGES) - 1) & 1);
                    if (!good) break;
                }
                uint8_t *st = smem + s * P::STAGE;
                const int t0 = (tile0 + i) * P::TT;
                tc::mbar_arrive_expect_tx(&gsfull[s], g_tx);
                tc::tma_load_2d(st + P::DU_OFF, &tmdu, 0, t0, &gsfull[s]);
                if (SG) {
                    for (int j = 0; j < N; ++j)
                        tc::tma_load_2d(st + P::G_OFF + j * P::XBOX, &tmg,
                                        int(int64_t(j) * C + c0), t0, &gsfull[s]);
                    tc::tma_load_2d(st + P::Y_OFF, &tmy, int(c0), t0, &gsfull[s]);
                }
                gissued = i + 1;
            }
            if (i >= P::STAGES) {
                // n = 8: tile i - 2's dx out; then x is free once the MMAs
                // (n = 4: and the epilogue) are done with it
                if (P::STORER) {
                    good = store_dx(i - P::STAGES);
                    if (!good) break;
                    stored = i - P::STAGES + 1;
                    if (lane < N) tc::bulk_wait_read_all();
                    __syncwarp();
                }
                good = lane0_wait(&empty[s], ((i / P::STAGES) - 1) & 1);
                if (!good) break;
            }
            if (lane == 0) {
                uint8_t *st = smem + s * P::STAGE;
                const int t0 = (tile0 + i) * P::TT;
                tc::mbar_arrive_expect_tx(&full[s], x_tx);
                for (int j = 0; j < N; ++j)
                    tc::tma_load_2d(st + j * P::XBOX, &tmx, int(int64_t(j) * C + c0), t0, &full[s]);
            }
            issued = i + 1;
        }
        if (P::STORER) {
            // the last tiles' dx
            for (int k = stored; good && k < issued; ++k) good = store_dx(k);
            if (lane < N) tc::bulk_wait_all();
        }
        // nothing may still be landing in shared memory when the CTA exits
        if (lane == 0)
            for (int i = max(0, issued - P::STAGES); i < issued; ++i) {
                tc::mbar_wait(&full[i % P::STAGES], (i / P::STAGES) & 1, a.fault,
                              tc::kFaultTimeoutMisc);
            }
        if (P::SPLIT && lane == 0)
            for (int i = max(0, gissued - P::STAGES); i < gissued; ++i)
                tc::mbar_wait(&gsfull[i % P::STAGES], (i / P::STAGES) & 1, a.fault,
                              tc::kFaultTimeoutMisc);
    } else if (P::NPRE == 3 && warp == 2) {
        // ------------------------------------- single-buffer producer (n = 8)
        // each buffer is refilled once the previous tile is done with it:
        // du_hl after the tile's MMAs, the per-token inputs and dout/dy after
        // the epilogue has read them
        if (lane == 0) {
            tc::tma_prefetch_desc(&tmdu);
            tc::tma_prefetch_desc(&tmdu2);
            if (TP) {
                tc::tma_prefetch_desc(&tmhres);
                tc::tma_prefetch_desc(&tmhpre);
                tc::tma_prefetch_desc(&tmhpost);
            }
            if (G1) {
                tc::tma_prefetch_desc(&tmg);
                tc::tma_prefetch_desc(&tmy);
            }
            uint8_t *par = smem + P::PAR_OFF;
            uint8_t *du1 = smem + P::DU1_OFF;
            uint8_t *g1 = smem + P::G1_OFF;
            int n1 = 0;   // tiles whose loads were issued
            for (int i = 0; i < ntiles && !*abort_v; ++i) {
                const int t0 = (tile0 + i) * P::TT;
                if (i >= 1 &&
                    !tc::mbar_wait(&duempty, (i - 1) & 1, a.fault, tc::kFaultTimeoutEmpty)) {
                    *abort_v = 1;
                    break;
                }
                tc::mbar_arrive_expect_tx(&dufull, P::DU_BYTES);
                for (int u = 0; u < P::DU_ATOMS; ++u)
                    tc::tma_load_2d(du1 + u * P::DU_ATOM_BYTES, &tmdu, u * 64, t0, &dufull);
                tc::tma_load_2d(du1 + P::DU_TAIL, &tmdu2, 128, t0, &dufull);
                if (G1) {
                    if (i >= 1 &&
                        !tc::mbar_wait(&gempty, (i - 1) & 1, a.fault, tc::kFaultTimeoutEmpty)) {
                        *abort_v = 1;
                        break;
                    }
                    tc::mbar_arrive_expect_tx(&gfull, P::G1_BYTES);
                    for (int j = 0; j < N; ++j)
                        tc::tma_load_2d(g1 + j * P::XBOX, &tmg, int(int64_t(j) * C + c0), t0,
                                        &gfull);
                    tc::tma_load_2d(g1 + N * P::XBOX, &tmy, int(c0), t0, &gfull);
                }
                if (TP) {
                    if (i >= 1 &&
                        !tc::mbar_wait(&pempty, (i - 1) & 1, a.fault, tc::kFaultTimeoutEmpty)) {
                        *abort_v = 1;
                        break;
                    }
                    tc::mbar_arrive_expect_tx(&pfull, P::PAR_BYTES);
                    tc::tma_load_2d(par, &tmhres, 0, t0, &pfull);
                    tc::tma_load_2d(par + P::TT * 128, &tmhres, 32, t0, &pfull);
                    tc::tma_load_2d(par + P::PH_PRE, &tmhpre, 0, t0, &pfull);
                    tc::tma_load_2d(par + P::PH_POST, &tmhpost, 0, t0, &pfull);
                }
                n1 = i + 1;
            }
            if (n1 > 0) {
                tc::mbar_wait(&dufull, (n1 - 1) & 1, a.fault, tc::kFaultTimeoutMisc);
                if (TP) tc::mbar_wait(&pfull, (n1 - 1) & 1, a.fault, tc::kFaultTimeoutMisc);
                if (G1) tc::mbar_wait(&gfull, (n1 - 1) & 1, a.fault, tc::kFaultTimeoutMisc);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issue
        if (lane == 0) {
            constexpr uint32_t idesc_dx = tc::idesc_bf16_f32(128, 128, 0, 0);
            constexpr uint32_t idesc_dw = tc::idesc_bf16_f32(128, P::NW, 1, 1);
            bool ok = tc::mbar_wait(&wfull, 0, a.fault, tc::kFaultTimeoutFull);
            const uint32_t wb = tc::smem_u32(wtile);
            for (int i = 0; ok && i < ntiles; ++i) {
                const int s = i % P::STAGES, b = i & 1;
                // du_hl (n = 4: the stage's G part) before the dx GEMM; x later
                if (*abort_v ||
                    (N == 4 && !tc::mbar_wait(&gsfull[s], (i / P::STAGES) & 1, a.fault,
                                              tc::kFaultTimeoutFull)) ||
                    (N == 8 && !tc::mbar_wait(&dufull, i & 1, a.fault, tc::kFaultTimeoutFull))) {
                    ok = false;
                    break;
                }
                tc::tc_fence_after();
                const uint32_t xs = tc::smem_u32(smem + s * P::STAGE);
                const uint32_t dus = N == 4 ? xs + P::DU_OFF : tc::smem_u32(smem + P::DU1_OFF);
                // dx accumulator b must have been drained by the epilogue (tile i-2)
                if (i >= 2 &&
                    !tc::mbar_wait(&d2empty[b], ((i >> 1) - 1) & 1, a.fault, tc::kFaultTimeoutAcc)) {
                    ok = false;
                    break;
                }
                tc::tc_fence_after();
                // K steps: du_hl[0,2O) against [W_hi | W_hi], then du_hi against W_lo
#pragma unroll
                for (int kk = 0; kk < P::KSTEP_A + P::KSTEP_B; ++kk) {
                    const int acol = kk < P::KSTEP_A ? 16 * kk : 16 * (kk - P::KSTEP_A);
                    uint64_t ad, bd;
                    if (N == 4) {
                        const int bcol = 16 * kk;
                        ad = tc::make_desc(dus + (acol / 64) * P::DU_ATOM_BYTES + (acol % 64) * 2, 16,
                                           1024, tc::kSwz128);
                        bd = tc::make_desc(wb + (bcol / 64) * P::W_PLANE_BYTES + (bcol % 64) * 2, 16,
                                           1024, tc::kSwz128);
                    } else {
                        // du columns [0,128) in the two atoms, [128,160) in the tail
                        ad = acol < 128 ? tc::make_desc(dus + (acol / 64) * P::DU_ATOM_BYTES +
                                                            (acol % 64) * 2,
                                                        16, 1024, tc::kSwz128)
                                        : tc::make_desc(dus + P::DU_TAIL + (acol - 128) * 2, 16,
                                                        512, tc::kSwz64);
                        // W step m of W_hi (kk < KSTEP_A) or W_lo
                        const int lo = kk < P::KSTEP_A ? 0 : 1;
                        const int m = kk < P::KSTEP_A ? kk % P::KSTEP_B : kk - P::KSTEP_A;
                        bd = m < 4 ? tc::make_desc(wb + lo * P::W_PLANE_BYTES + m * 32, 16, 1024,
                                                   tc::kSwz128)
                                   : tc::make_desc(wb + P::W_TAIL + lo * 32, 16, 512, tc::kSwz64);
                    }
                    tc::mma_bf16(tmem + P::D2_COL + b * 128, ad, bd, idesc_dx, kk > 0 ? 1u : 0u);
                }
                tc::mma_commit(&d2full[b]);
                if (!tc::mbar_wait(&full[s], (i / P::STAGES) & 1, a.fault, tc::kFaultTimeoutFull)) {
                    ok = false;
                    break;
                }
                tc::tc_fence_after();
                // dW += x^T du_hl over the tile's 128 tokens, 16 per step
#pragma unroll
                for (int ks = 0; ks < P::TT / 16; ++ks) {
                    const uint64_t ad =
                        tc::make_desc(xs + ks * 16 * P::XROW, P::XBOX, 8 * P::XROW, P::XSWZ);
                    const uint32_t acc = (i > 0 || ks > 0) ? 1u : 0u;
                    if (N == 4) {
                        const uint64_t bd =
                            tc::make_desc(dus + ks * 16 * 128, P::DU_ATOM_BYTES, 1024, tc::kSwz128);
                        tc::mma_bf16(tmem + P::D1_COL, ad, bd, idesc_dw, acc);
                    } else {
                        // du columns [0,128) (N = 128) and the tail [128,160) (N = 32)
                        constexpr uint32_t idesc_dw1 = tc::idesc_bf16_f32(128, 128, 1, 1);
                        constexpr uint32_t idesc_dw2 = tc::idesc_bf16_f32(128, 32, 1, 1);
                        const uint64_t bd1 =
                            tc::make_desc(dus + ks * 16 * 128, P::DU_ATOM_BYTES, 1024, tc::kSwz128);
                        const uint64_t bd2 = tc::make_desc(dus + P::DU_TAIL + ks * 16 * 64,
                                                           P::DU_TAIL_BYTES, 512, tc::kSwz64);
                        tc::mma_bf16(tmem + P::D1_COL, ad, bd1, idesc_dw1, acc);
                        tc::mma_bf16(tmem + P::D1_COL + 128, ad, bd2, idesc_dw2, acc);
                    }
                }
                tc::mma_commit(&xfree[s]);
                if (P::SPLIT) tc::mma_commit(&empty[s]);
                if (SG) {
                    // dbias: dout^T [du_hl | H_post hi | H_post lo] over the tile
                    constexpr uint32_t idesc_db = tc::idesc_bf16_f32(128, P::D3_N, 1, 1);
#pragma unroll
                    for (int ks = 0; ks < P::TT / 16; ++ks) {
                        const uint64_t ad = tc::make_desc(xs + P::G_OFF + ks * 16 * P::XROW,
                                                          P::XBOX, 8 * P::XROW, P::XSWZ);
                        const uint64_t bd = tc::make_desc(dus + ks * 16 * 128, P::DU_ATOM_BYTES,
                                                          1024, tc::kSwz128);
                        tc::mma_bf16(tmem + P::D3_COL, ad, bd, idesc_db,
                                     (i > 0 || ks > 0) ? 1u : 0u);
                    }
                }
                if (P::SPLIT)
                    tc::mma_commit(&gsempty[s]);
                else
                    tc::mma_commit(&empty[s]);
                if (N == 8) tc::mma_commit(&duempty);
            }
            if (!ok) *abort_v = 1;
            tc::mma_commit(&d1full);
            tc::mbar_wait(&d1full, 0, a.fault, tc::kFaultTimeoutAcc);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        // The W tile of this slice in the swizzled K-major layout of the MMA B
        // operand (16-byte chunk q of row rr at rr*128 + ((q ^ (rr % 8)) * 16)
        // in a 128-byte plane, at rr*64 + ((q ^ ((rr / 2) % 4)) * 16) in the
        // 64-byte tail); rows past C are zero.  n = 4: [W_hi | W_hi | W_lo | 0]
        // in 64-column planes.  n = 8: W_hi [0,64), W_lo [0,64), and the tail
        // [W_hi [64,80) | W_lo [64,80)].
        constexpr int W_CHUNKS = P::W_PLANES * 128 * 8 + (N == 8 ? 128 * 4 : 0);
        float wmax = 0.f;   // max |W| of the values this thread loads
        for (int idx = threadIdx.x - 32 * P::NPRE; idx < W_CHUNKS; idx += 32 * P::EPI_WARPS) {
            int rr, col;
            bool lo;
            uint32_t dst;
            if (idx < P::W_PLANES * 128 * 8) {
                const int p = idx >> 10, qc = idx & 7;
                rr = (idx >> 3) & 127;
                col = N == 4 ? p * 64 + qc * 8 : qc * 8;
                lo = N == 4 ? col >= 2 * O : p == 1;
                dst = tc::smem_u32(wtile + p * P::W_PLANE_BYTES + rr * 128 + ((qc ^ (rr & 7)) << 4));
            } else {
                const int j = idx - P::W_PLANES * 128 * 8, qc = j & 3;
                rr = j >> 2;
                col = 64 + (qc & 1) * 8;
                lo = qc >= 2;
                dst = tc::smem_u32(wtile + P::W_TAIL + rr * 64 + ((qc ^ ((rr >> 1) & 3)) << 4));
            }
            const int64_t cw = c0 + rr % CW;
            float w[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            if ((N == 8 || col < 3 * O) && cw < C) {
                const float4 *src = reinterpret_cast<const float4 *>(
                    a.W + (int64_t(rr / CW) * C + cw) * O + col % O);
                const float4 v0 = __ldg(src), v1 = __ldg(src + 1);
                w[0] = v0.x; w[1] = v0.y; w[2] = v0.z; w[3] = v0.w;
                w[4] = v1.x; w[5] = v1.y; w[6] = v1.z; w[7] = v1.w;
#pragma unroll
                for (int e = 0; e < 8; ++e) wmax = fmaxf(wmax, fabsf(w[e]));
                if (lo)
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        w[e] -= __bfloat162float(__float2bfloat16_rn(w[e]));
            }
            const uint4 v = pack8(w);
            asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(dst), "r"(v.x), "r"(v.y),
                         "r"(v.z), "r"(v.w)
                         : "memory");
        }
        tc::fence_proxy_async_smem();
        // the slice's max |W|: each warp folds its maximum in before its
        // threads report their part of the W tile on the W barrier, and every
        // epilogue thread reads the total once that barrier has completed
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) wmax = fmaxf(wmax, __shfl_xor_sync(kFull, wmax, m));
        if (lane == 0) atomicMax(&wmax_bits, __float_as_uint(wmax));
        tc::mbar_release(&wfull);
        if (!tc::mbar_wait(&wfull, 0, a.fault, tc::kFaultTimeoutMisc)) *abort_v = 1;
        // a token whose sum_o |du_o| times this bound factor exceeds
        // kExactAbove takes the exact path
        const float wbound = __uint_as_float(wmax_bits) * kSplitBound;

        const int q = warp & 3;              // TMEM lane quadrant
        const int h = (warp - P::NPRE) >> 2; // this thread's 8-channel chunk of every stream
        const int r = q * 32 + lane;         // token row in the tile / k row of dW
        const uint32_t trow = tmem + (uint32_t(q * 32) << 16);
        const int64_t cc = c0 + h * 8;       // first channel of the chunk
        const bool cvalid = cc < C;          // the last slice may pass C
        float bias_acc = 0.f;                // lane l: running total of channel cc + (l % 8)
        f32x2 dfacc[4] = {0ull, 0ull, 0ull, 0ull};
        bool ok = true;
        // The four warps of a quadrant share its 32 token rows: together they
        // copy the rows' inputs of a tile into shared memory one tile ahead
        // (H_res chunk h, H_pre by h = 0, coef by one warp; rows past T are
        // zero-filled) and meet at a named barrier before and after reading.
        const uint32_t prow = tc::smem_u32(smem + P::PAR_OFF) + r * P::PAR_ROW;
        const uint32_t pcoef = tc::smem_u32(smem + P::PAR_OFF + P::TT * P::PAR_ROW) + r * 4;
        const uint32_t pdub = pcoef + P::TT * 4;
        auto stage_params = [&](int tile) {
            const int64_t tp = int64_t(tile) * P::TT + r;
            const bool v = tp < a.T;
            const int64_t tv = v ? tp : 0;
            if (LAYER) {
                tc::cp_async16(prow + h * 16, a.Hres + tv * N * N + h * 4, v ? 16u : 0u);
                if (h == 0) tc::cp_async16(prow + 64, a.Hpre + tv * N, v ? 16u : 0u);
            }
            if (h == (LAYER ? 1 : 0)) {
                tc::cp_async4(pcoef, a.coef + tv, v ? 4u : 0u);
                tc::cp_async4(pdub, a.dub + tv, v ? 4u : 0u);
            }
            tc::cp_async_commit();
        };
        if (P::STAGE_P && ntiles > 0) stage_params(tile0);
        // n = 8: coef and sum |du| of a tile are loaded one tile ahead (a load
        // issued at the tile's start comes back from L2 after its first use)
        float coef_nx = 0.f, dub_nx = 0.f;
        if (!P::STAGE_P && ntiles > 0 && int64_t(tile0) * P::TT + r < a.T) {
            coef_nx = __ldg(a.coef + int64_t(tile0) * P::TT + r);
            dub_nx = __ldg(a.dub + int64_t(tile0) * P::TT + r);
        }
        for (int i = 0; i < ntiles; ++i) {
            const int s = i % P::STAGES, b = i & 1;
            const int64_t t = int64_t(tile0 + i) * P::TT + r;
            const bool valid = t < a.T;
            // per-token inputs, fetched before waiting on the tensor cores
            float coef = 0.f, dub = 0.f, hpre[N], hpost[N], hres[LAYER ? N * N : 1];
#pragma unroll
            for (int j = 0; j < N; ++j) hpre[j] = hpost[j] = 0.f;
#pragma unroll
            for (int e = 0; e < (LAYER ? N * N : 1); ++e) hres[e] = 0.f;
            uint4 g[N], gy = make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int ii = 0; ii < N; ++ii) g[ii] = make_uint4(0, 0, 0, 0);
            if (P::STAGE_P) {
                // every warp of the quadrant passes both barriers on every
                // tile, also after a failure, so none of them waits alone
                tc::cp_async_wait_all();
                tc::named_bar_sync(1 + q, 128);
                if (LAYER) {
#pragma unroll
                    for (int e = 0; e < N * N; e += 4) {
                        const uint4 v = lds128(prow + e * 4);
                        hres[e] = __uint_as_float(v.x);
                        hres[e + 1] = __uint_as_float(v.y);
                        hres[e + 2] = __uint_as_float(v.z);
                        hres[e + 3] = __uint_as_float(v.w);
                    }
                    const uint4 v = lds128(prow + 64);
                    hpre[0] = __uint_as_float(v.x);
                    hpre[1] = __uint_as_float(v.y);
                    hpre[2] = __uint_as_float(v.z);
                    hpre[3] = __uint_as_float(v.w);
                }
                coef = lds32f(pcoef);
                dub = lds32f(pdub);
                tc::named_bar_sync(1 + q, 128);
                if (i + 1 < ntiles) stage_params(tile0 + i + 1);
                if (!ok) continue;
            } else {
                coef = coef_nx;
                dub = dub_nx;
                coef_nx = dub_nx = 0.f;
                if (i + 1 < ntiles && t + P::TT < a.T) {
                    coef_nx = __ldg(a.coef + t + P::TT);
                    dub_nx = __ldg(a.dub + t + P::TT);
                }
                if (valid) {
                    if (LAYER && !TP) {
#pragma unroll
                        for (int j = 0; j < N; ++j) {
                            hpre[j] = __ldg(a.Hpre + t * N + j);
                            hpost[j] = __ldg(a.Hpost + t * N + j);
                        }
#pragma unroll
                        for (int e = 0; e < N * N; e += 4) {
                            const float4 v =
                                __ldg(reinterpret_cast<const float4 *>(a.Hres + t * N * N + e));
                            hres[e] = v.x;
                            hres[e + 1] = v.y;
                            hres[e + 2] = v.z;
                            hres[e + 3] = v.w;
                        }
                    }
                }
                if (TP) {
                    // this tile's H_res, H_pre and H_post rows from the TMA
                    // boxes (rows past T read as zero), then the buffer goes
                    // back to the producer for the next tile
                    if (*abort_v || !tc::mbar_wait(&pfull, i & 1, a.fault, tc::kFaultTimeoutFull)) {
                        ok = false;
                        break;
                    }
                    const uint32_t pb = tc::smem_u32(smem + P::PAR_OFF);
#pragma unroll
                    for (int c4 = 0; c4 < N / 4; ++c4) {
                        const uint32_t off = r * 32 + ((c4 ^ ((r >> 2) & 1)) << 4);
                        const uint4 vp = lds128(pb + P::PH_PRE + off);
                        const uint4 vq = lds128(pb + P::PH_POST + off);
                        hpre[4 * c4] = __uint_as_float(vp.x);
                        hpre[4 * c4 + 1] = __uint_as_float(vp.y);
                        hpre[4 * c4 + 2] = __uint_as_float(vp.z);
                        hpre[4 * c4 + 3] = __uint_as_float(vp.w);
                        hpost[4 * c4] = __uint_as_float(vq.x);
                        hpost[4 * c4 + 1] = __uint_as_float(vq.y);
                        hpost[4 * c4 + 2] = __uint_as_float(vq.z);
                        hpost[4 * c4 + 3] = __uint_as_float(vq.w);
                    }
                }
                if (G1) {
                    // dout and dy of this tile (rows past T read as zero;
                    // chunks past C are read but never stored)
                    if (*abort_v || !tc::mbar_wait(&gfull, i & 1, a.fault, tc::kFaultTimeoutFull)) {
                        ok = false;
                        break;
                    }
                    const uint8_t *gb = smem + P::G1_OFF;
#pragma unroll
                    for (int ii = 0; ii < N; ++ii) g[ii] = box_chunk<N>(gb + ii * P::XBOX, r, h);
                    gy = box_chunk<N>(gb + N * P::XBOX, r, h);
                    tc::mbar_release(&gempty);
                }
            }
            // `bar` (n = 4: the stage's G part; n = 8: x) and the dx accumulator
            // of this tile; then the exact path (rare: rows of near-zero RMS):
            // a warp with such a token rewrites that token's dx_gemm values in
            // TMEM with du.W^T from the fp32 values before the usual reads below
            auto part_and_acc = [&](uint64_t *bar) -> bool {
                if (*abort_v ||
                    !tc::mbar_wait(bar, (i / P::STAGES) & 1, a.fault, tc::kFaultTimeoutFull) ||
                    !tc::mbar_wait(&d2full[b], (i >> 1) & 1, a.fault, tc::kFaultTimeoutAcc))
                    return false;
                tc::tc_fence_after();
                const bool exact = valid && cvalid && dub * wbound > kExactAbove;
                if (__any_sync(kFull, exact)) {
                    const uint32_t tb = trow + P::D2_COL + b * 128 + h * 8;
#pragma unroll 1
                    for (int j = 0; j < N; ++j) {
                        float v[8];
                        tc::tmem_ld8_wait(tb + j * CW, v);
                        if (exact) {
                            const float *wrow = a.W + (int64_t(j) * C + cc) * O;
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                v[e] = exact_du_w(a.du32 + t * O, wrow + e * O, O);
                        }
                        __syncwarp();
                        tc::tmem_st8_wait(tb + j * CW, v);
                    }
                }
                return true;
            };
            // n = 4: dout and dy (the G part) and the accumulator before the mix
            if (P::SPLIT && !part_and_acc(&gsfull[s])) {
                ok = false;
                if (P::STAGE_P) continue;
                break;
            }
            const uint8_t *st = smem + s * P::STAGE;
            // (releasing the stage right after these reads, before the
            // arithmetic, measured slower: the stage goes back at the end)
            uint4 xr[N];
            if (SG) {
#pragma unroll
                for (int ii = 0; ii < N; ++ii) g[ii] = box_chunk<N>(st + P::G_OFF + ii * P::XBOX, r, h);
                gy = box_chunk<N>(st + P::Y_OFF, r, h);
            }
            // mix[j][e] = H_pre[j] dy[e] + sum_i H_res[j][i] dout_i[e];  df = sum_i H_post[i] dout_i
            // (element pairs in f32x2 arithmetic)
            f32x2 mix[LAYER ? N : 1][4];
            if (LAYER) {
                f32x2 gyv[4];
                unpack8x2(gy, gyv);
#pragma unroll
                for (int j = 0; j < N; ++j) {
                    const f32x2 w2 = f2_make(hpre[j], hpre[j]);
#pragma unroll
                    for (int p = 0; p < 4; ++p) mix[j][p] = f2_mul(w2, gyv[p]);
                }
#pragma unroll
                for (int ii = 0; ii < N; ++ii) {
                    f32x2 dv[4];
                    unpack8x2(g[ii], dv);
                    if (!SG) {
                        const f32x2 w2 = f2_make(hpost[ii], hpost[ii]);
#pragma unroll
                        for (int p = 0; p < 4; ++p) dfacc[p] = f2_fma(w2, dv[p], dfacc[p]);
                    }
                    // n = 8: the parameter buffer holds H_res transposed, so
                    // H_res[t][0..8)[ii] are two 16-byte chunks of row ii of
                    // HresT (128-byte-swizzled rows of 32 floats)
                    float hcol[N];
                    if (TP) {
                        const uint32_t pb = tc::smem_u32(smem + P::PAR_OFF) +
                                            ((ii * N) >> 5) * (P::TT * 128) + r * 128;
#pragma unroll
                        for (int c4 = 0; c4 < N / 4; ++c4) {
                            const int chunk = (((ii * N) & 31) >> 2) + c4;
                            const uint4 v = lds128(pb + ((chunk ^ (r & 7)) << 4));
                            hcol[4 * c4] = __uint_as_float(v.x);
                            hcol[4 * c4 + 1] = __uint_as_float(v.y);
                            hcol[4 * c4 + 2] = __uint_as_float(v.z);
                            hcol[4 * c4 + 3] = __uint_as_float(v.w);
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < N; ++j) hcol[j] = hres[j * N + ii];
                    }
#pragma unroll
                    for (int j = 0; j < N; ++j) {
                        const f32x2 w2 = f2_make(hcol[j], hcol[j]);
#pragma unroll
                        for (int p = 0; p < 4; ++p) mix[j][p] = f2_fma(w2, dv[p], mix[j][p]);
                    }
                }
                if (TP) {
                    // this thread has read the parameter buffer
                    tc::mbar_release(&pempty);
                }
                if (P::SPLIT) {
                    // n = 4: dout and dy have been read; the G part goes back
                    // once the tile's MMAs are done with it too
                    tc::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(&gsempty[s]);
                }
            }
            // dx_gemm of this chunk for every stream: all TMEM loads, one wait
            constexpr int JB = 2;  // streams per batch of TMEM loads
            const f32x2 coef2 = f2_make(coef, coef);
            // x (n = 8: with the accumulator)
            if (P::SPLIT ? (*abort_v || !tc::mbar_wait(&full[s], (i / P::STAGES) & 1, a.fault,
                                                        tc::kFaultTimeoutFull))
                         : !part_and_acc(&full[s])) {
                ok = false;
                if (P::STAGE_P) continue;
                break;
            }
            // dx overwrites x in the stage (the stream boxes have dx's layout:
            // each thread writes the chunk it has just read) once the tile's
            // dW MMAs have read it
            if (*abort_v ||
                !tc::mbar_wait(&xfree[s], (i / P::STAGES) & 1, a.fault, tc::kFaultTimeoutAcc)) {
                ok = false;
                if (P::STAGE_P) continue;
                break;
            }
#pragma unroll
            for (int j0 = 0; j0 < N; j0 += JB) {
                float acc[JB][8];
                static_assert(JB == 2, "two TMEM loads per batch");
                const uint32_t ta = trow + P::D2_COL + b * 128 + j0 * CW + h * 8;
                tc::tmem_ld8x2_wait(ta, ta + CW, acc[0], acc[1]);
#pragma unroll
                for (int jj = 0; jj < JB; ++jj) xr[j0 + jj] = box_chunk<N>(st + (j0 + jj) * P::XBOX, r, h);
#pragma unroll
                for (int jj = 0; jj < JB; ++jj) {
                    const int j = j0 + jj;
                    f32x2 xv[4], o[4];
                    unpack8x2(xr[j], xv);
#pragma unroll
                    for (int p = 0; p < 4; ++p) {
                        o[p] = f2_fma(coef2, xv[p], f2_make(acc[jj][2 * p], acc[jj][2 * p + 1]));
                        if (LAYER) o[p] = f2_add(o[p], mix[j][p]);
                    }
                    const uint4 v = pack8x2(o);
                    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(
                                     box_chunk_addr<N>(st + j * P::XBOX, r, h)),
                                 "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                                 : "memory");
                }
            }
            // this thread is done with the stage and its dx chunks are there
            // (visible to the TMA engine).  n = 8: the stage producer stores
            // them once every thread's are.  n = 4: lane j of the quadrant's
            // chunk-0 warp stores stream j's 32 rows once the quadrant's are,
            // and the warp releases the stage after the stores have read it.
            // D2 buffer b has been read.
            tc::fence_proxy_async_smem();
            if (P::STORER) {
                tc::mbar_arrive(&dxfull[s][0]);
            } else {
                tc::mbar_arrive(&dxfull[s][q]);
                if (h == 0 && lane < N) {
                    if (tc::mbar_wait(&dxfull[s][q], (i / P::STAGES) & 1, a.fault,
                                      tc::kFaultTimeoutFull)) {
                        const int z = (tile0 + i) * P::TT + q * 32;
                        if (z < a.T) {
                            tc::tma_store_3d(&tmdx, st + lane * P::XBOX + q * 32 * P::XROW, int(c0),
                                             lane, z);
                            tc::bulk_commit_group();
                            tc::bulk_wait_read_all();
                        }
                    } else {
                        *abort_v = 1;
                    }
                }
            }
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (!P::STORER) tc::mbar_arrive(&empty[s]);
                tc::mbar_arrive(&d2empty[b]);
            }
        }
        if (P::STAGE_P) tc::cp_async_wait_all();
        // (n = 4) the dx stores are complete before the CTA exits
        if (!P::STORER && h == 0 && lane < N) tc::bulk_wait_all();
        if (!ok) *abort_v = 1;
        // dW partial of this split: D1 rows are the 128 k of the slice; the
        // chunk-0 warps write it
        const bool krow = c0 + (r % CW) < C;  // dW row exists
        if (ok && h == 0 && tc::mbar_wait(&d1full, 0, a.fault, tc::kFaultTimeoutAcc)) {
            tc::tc_fence_after();
            const int j = r / CW, c = r % CW;
            float *dst = a.dWpart + (int64_t(split) * K + int64_t(j) * C + c0 + c) * O;
            if (O == 24) {
                float v[48];
#pragma unroll
                for (int m = 0; m < 3; ++m) {
                    float w16[16];
                    tc::tmem_ld16_wait(trow + P::D1_COL + m * 16, w16);
#pragma unroll
                    for (int e = 0; e < 16; ++e) v[m * 16 + e] = w16[e];
                }
#pragma unroll
                for (int o4 = 0; o4 < O / 4; ++o4)
                    if (krow)
                        reinterpret_cast<float4 *>(dst)[o4] = make_float4(
                            v[4 * o4] + v[O + 4 * o4], v[4 * o4 + 1] + v[O + 4 * o4 + 1],
                            v[4 * o4 + 2] + v[O + 4 * o4 + 2], v[4 * o4 + 3] + v[O + 4 * o4 + 3]);
            } else {
#pragma unroll 1
                for (int m = 0; m < O / 16; ++m) {
                    float hi[16], lo[16];
                    tc::tmem_ld16x2_wait(trow + P::D1_COL + m * 16, trow + P::D1_COL + O + m * 16,
                                         hi, lo);
#pragma unroll
                    for (int o4 = 0; o4 < 4; ++o4)
                        if (krow)
                            reinterpret_cast<float4 *>(dst + m * 16)[o4] = make_float4(
                                hi[4 * o4] + lo[4 * o4], hi[4 * o4 + 1] + lo[4 * o4 + 1],
                                hi[4 * o4 + 2] + lo[4 * o4 + 2], hi[4 * o4 + 3] + lo[4 * o4 + 3]);
                }
            }
        }
        if (LAYER && !SG) {
            float dfs[8];
#pragma unroll
            for (int p = 0; p < 4; ++p) f2_split(dfacc[p], dfs[2 * p], dfs[2 * p + 1]);
            bias_acc = warp_column_sum<8>(dfs);
        }
        if (LAYER && !SG && lane < 8) bias_red[q][h * 8 + lane] = bias_acc;
        if (SG && h == 0) {
            // D3 row r is k = stream q, channel lane: its dbias term is the
            // stream's H_post column pair
            float v = 0.f;
            if (ok) {
                float d3[16];
                tc::tmem_ld16_wait(trow + P::D3_COL + 2 * O, d3);
#pragma unroll
                for (int e = 0; e < N; ++e)
                    if (e == q) v = d3[e] + d3[N + e];
            }
            bias_red[q][lane] = v;
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    if (LAYER && threadIdx.x < CW && c0 + threadIdx.x < C && !abort_flag) {
        const float v = bias_red[0][threadIdx.x] + bias_red[1][threadIdx.x] +
                        bias_red[2][threadIdx.x] + bias_red[3][threadIdx.x];
        a.dbiaspart[int64_t(split) * C + c0 + threadIdx.x] = v;
    }
    if (warp == 1) tc::tmem_dealloc(tmem, P::TMEM_COLS);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
int bwd_tc_du_cols(int n) { return n == 4 ? BwdTc<4>::DU_COLS : BwdTc<8>::DU_COLS; }

int bwd_tc_splits(int64_t T, int n, int64_t C)
{
    const int64_t slices = (C + 128 / n - 1) / (128 / n);
    const int64_t tiles = (T + 127) / 128;
    int64_t s = int64_t(kSplitSms) / (slices > 0 ? slices : 1);
    if (s < 1) s = 1;
    if (s > tiles) s = tiles;
    if (s > 8) s = 8;
    return int(s);
}

template <int N, bool LAYER>
static cudaError_t bwd_tc_impl(const bf16 *x, const bf16 *du_hl, const BwdTcArgs &args,
                               int splits, cudaStream_t s)
{
    using P = BwdTc<N>;
    const int64_t T = args.T, C = args.C, K = int64_t(N) * C;
    CUtensorMap tmx, tmdu, tmg, tmy, tmdu2, tmhres, tmhpre, tmhpost, tmdx;
    const CUtensorMapSwizzle xsw = N == 4 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B;
    if (!tmap_bf16_2d(&tmx, x, uint64_t(T), uint64_t(K), P::TT, P::CW, xsw) ||
        !tmap_bf16_2d(&tmdu, du_hl, uint64_t(T), uint64_t(P::DU_COLS), P::TT, 64,
               CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    tmg = tmy = tmdu2 = tmhres = tmhpre = tmhpost = tmdx = tmx;
    {
        // dx as [T][n][C]: a stream's box of the slice's channels over a tile
        // (n = 8) or a quadrant's 32 tokens (n = 4)
        const uint64_t dims[3] = {uint64_t(C), uint64_t(N), uint64_t(T)};
        const uint64_t strides[2] = {uint64_t(C) * 2, uint64_t(C) * 2 * N};
        const uint32_t box[3] = {uint32_t(P::CW), 1, P::STORER ? uint32_t(P::TT) : 32u};
        if (!tmap_bf16(&tmdx, args.dx, 3, dims, strides, box, xsw)) return cudaErrorInvalidValue;
    }
    if (LAYER) {
        if (!tmap_bf16_2d(&tmg, args.dout, uint64_t(T), uint64_t(K), P::TT, P::CW, xsw) ||
            !tmap_bf16_2d(&tmy, args.dy, uint64_t(T), uint64_t(C), P::TT, P::CW, xsw))
            return cudaErrorInvalidValue;
    }
    if (N == 8 && !tmap_bf16_2d(&tmdu2, du_hl, uint64_t(T), uint64_t(P::DU_COLS), P::TT, 32,
                                CU_TENSOR_MAP_SWIZZLE_64B))
        return cudaErrorInvalidValue;
    if (LAYER && P::TMA_P) {
        if (!tmap_f32_2d(&tmhres, args.Hres, uint64_t(T), uint64_t(N * N), P::TT, 32,
                         CU_TENSOR_MAP_SWIZZLE_128B) ||
            !tmap_f32_2d(&tmhpre, args.Hpre, uint64_t(T), uint64_t(N), P::TT, 8,
                         CU_TENSOR_MAP_SWIZZLE_32B) ||
            !tmap_f32_2d(&tmhpost, args.Hpost, uint64_t(T), uint64_t(N), P::TT, 8,
                         CU_TENSOR_MAP_SWIZZLE_32B))
            return cudaErrorInvalidValue;
    }
    cudaError_t e = set_smem_limit(reinterpret_cast<const void *>(k_bwd_tc<N, LAYER>), P::SMEM);
    if (e != cudaSuccess) return e;
    dim3 grid(unsigned((C + P::CW - 1) / P::CW), unsigned(splits));
    {
        MHC_PROF("k_bwd_tc", s);
        launch_k(k_bwd_tc<N, LAYER>, dim3(grid), dim3(P::THREADS), P::SMEM, s, tmx, tmdu, tmg, tmy,
                 tmdu2, tmhres, tmhpre, tmhpost, tmdx, args);
    }
    return cudaGetLastError();
}

cudaError_t launch_bwd_tc(const bf16 *x, const float *W, const bf16 *du_hl, const float *du32,
                          const float *dub, const float *coef, int64_t T, int n, int64_t C,
                          const bf16 *dout, const bf16 *dy, const float *Hpre, const float *Hres,
                          const float *Hpost, bf16 *dx, float *dWpart, float *dbiaspart,
                          int splits, int *fault, cudaStream_t s)
{
    BwdTcArgs a;
    a.W = W;
    a.du32 = du32;
    a.dub = dub;
    a.dout = dout;
    a.dy = dy;
    a.coef = coef;
    a.Hpre = Hpre;
    a.Hres = Hres;
    a.Hpost = Hpost;
    a.dx = dx;
    a.dWpart = dWpart;
    a.dbiaspart = dbiaspart;
    a.T = T;
    a.C = C;
    a.tiles_total = int((T + 127) / 128);
    a.tiles_per_split = (a.tiles_total + splits - 1) / splits;
    a.fault = fault;
    const bool layer = dout != nullptr;
    if (n == 4)
        return layer ? bwd_tc_impl<4, true>(x, du_hl, a, splits, s)
                     : bwd_tc_impl<4, false>(x, du_hl, a, splits, s);
    return layer ? bwd_tc_impl<8, true>(x, du_hl, a, splits, s)
                 : bwd_tc_impl<8, false>(x, du_hl, a, splits, s);
}

}  // namespace mhc
