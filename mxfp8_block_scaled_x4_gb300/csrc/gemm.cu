// gemm.cu -- MXFP8 block-scaled GEMM + padded-N slice + bias for sm_103a.
//
// Computes, for token rows i and output features j < N (vLLM PR #52204
// "[Kernel] Add FlashInfer TRTLLM MXFP8 linear backend", apply_weights: the
// mm_mxfp8 product with FP32 accumulation, then output[:, :N] + bias):
//   y[i][j] = bf16( sum_b 2^(sa[i,b]-127) 2^(sw[j,b]-127) sum_{k in b} qa[i,k] qw[j,k] + bias[j] )
//
// Orientation.  The weights are the MMA's A operand (M = 128 rows of N per
// tile) and the tokens its B operand (N = 16..256 tokens per tile): the
// accumulator D^T[n, token] lives in TMEM with one weight row per lane.  This
// is why N is padded to 128 and why the small-M case needs no padding of the
// token count beyond 16 (FlashInfer PR #1214, Highlights, makes the same
// choice: its MMA outputs come out transposed and are shuffled back).
//
// mxfp8_gemm_kernel<TT, PIPES, MODE> (TT tokens per tile, PIPES MMA
// pipelines per CTA, MODE plain / gated SwiGLU / 128x4 activation scales):
//   warp 0      TMA producer of pipe 0: per 128-wide K block, one 128x128
//               weight tile, the weight scales (one 512-byte bulk copy,
//               already in TMEM-copy order) and -- unless quantization is
//               fused -- the token tile (one TMA box) and its scales (the
//               raw 8x4 groups in one box, or the 128x4 tiles by bulk copy).
//   warp 1      TMEM allocator; its lane 0 alone is the MMA issuer of pipe 0:
//               copies both scale tiles into TMEM (tcgen05.cp 32x128b.warpx4),
//               issues four tcgen05.mma kind::mxf8f6f4 block_scale (K = 32
//               each) and commits the stage back to the producer.  Each
//               tcgen05/TMA/mbarrier instruction costs its issuing thread
//               ~55-170 cycles, which bounds one pipeline at small N.
//   warps 2..   epilogue (4 warps for TT = 32, else 8, one or two per TMEM
//               lane quadrant): tcgen05.ld, release the accumulator, then
//               + bias, BF16 rounding and masked stores (j < N, token < M);
//               the gated mode passes the up half to the gate half through
//               shared memory and stores silu(gate) * up.  With fused
//               quantization they first quantize the BF16 token rows of
//               each K block straight into the swizzled B tile and the
//               TMEM-copy scale order (same arithmetic as quant.cu).
//   next warp   8x4 scale re-order (unfused, 8x4 scales): token j of the
//               raw groups goes to word (j%32)*4 + (j%128)/32 of its
//               128-token chunk, the order tcgen05.cp 32x128b.warpx4 expects.
//   last warps  producers and MMA issuers of pipes 1..PIPES-1: pipe q takes
//               the local K blocks i with i % PIPES == q into its own stages
//               and its own TMEM accumulator; the epilogue sums the pipes'
//               accumulators in pipe order (deterministic).
// Schedules:
//   persistent   grid <= #SMs x occupancy, tiles strided over CTAs (large M,
//                grouped); a second TMEM accumulator per pipe where tensor
//                memory allows it, so the next tile's MMAs overlap this
//                tile's epilogue.
//   one tile     one output tile per cluster of `splits` CTAs, each a K range
//                (small M).  With splits > 1 each rank owns a slice of the
//                token columns; every rank stages its FP32 partials in its
//                idle pipeline stages and one bulk copy per peer moves the
//                peer's slice into the peer's shared memory, counted on the
//                peer's mbarrier; each owner sums its slice in rank order
//                (deterministic) as soon as its bytes have landed.
//   dual         mxfp8_gemm_dual_kernel<TT>: two 128-row weight tiles x 144,
//                160, 176 or 192 tokens per CTA tile (dense, large M), below.
// Programmatic dependent launch: the kernel lets the next grid start at once;
// it reads nothing a previous grid may write before griddepcontrol.wait,
// except the weights, their scales, the bias and the grouped offsets, which
// must be complete before the layer's first kernel may start.
// Every wait is bounded (4 s by default); a timeout sets g_gemm_error, every role
// unwinds, in-flight copies and MMAs are drained (again bounded), TMEM is
// freed and the kernel returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <atomic>

#include "debug_check.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "quant_block.cuh"

namespace mxk {

__device__ unsigned int g_gemm_error;

// Schedule of the last GEMM launch on the host (testing aid).
thread_local int t_last_schedule[5];
std::atomic<uint64_t> g_wait_limit_ns{0};  // testing hook, any thread; 0: kWaitNs

namespace {

constexpr uint64_t kWaitNs = 4000000000ull;   // default: 4 s per wait, then give up
constexpr uint64_t kDrainNs = 200000000ull;   // 0.2 s per drain wait
constexpr int kMaxExperts = 1024;

struct GemmArgs {
    CUtensorMap map_w;     // weights [experts*n_pad, k] u8, box {128, 128}, 128B swizzle
    CUtensorMap map_a;     // activations [m, k] u8, box {128, box_rows}, 128B swizzle
    CUtensorMap map_asf;   // 8x4 scales as [m8/8, k/4] u8, box {32, sf_groups}
    const uint8_t* wsf;
    const __nv_bfloat16* bias;
    __nv_bfloat16* y;
    const int32_t* offsets;  // grouped segment offsets, or null (dense)
    const __nv_bfloat16* x;  // fused quantization: BF16 activations [m, k], else null
    int m, n, n_pad, k, kq;  // kq = k / 128
    int experts, n_tiles;
    int box_rows, sf_groups;
    int stages, splits, persistent;
    const uint8_t* asf128;   // activation scales in the 128x4 layout (dense tiles of 128/256), or null
    int acc_bufs;            // TMEM accumulators per pipe: 2 lets tile t+1's MMAs overlap tile t's epilogue
    int num_tiles;           // dense (grouped counts tiles on the device)
    uint32_t tmem_cols;
    uint64_t wait_ns;        // limit of every pipeline wait
    uint8_t* hq;             // gated: h quantized to MXFP8 (E4M3 [m][n/2]) instead of BF16 y, or null
    uint8_t* hsf;            // gated: its 8x4 scales
};

template <int TT>
struct Geometry {
    static constexpr int kSfChunks = (TT + 127) / 128;          // 128-token scale chunks
    static constexpr int kOffW = 0;
    static constexpr int kOffA = 16384;
    static constexpr int kOffWsf = kOffA + TT * 128;
    static constexpr int kOffAsfRaw = kOffWsf + 512;
    static constexpr int kOffAsfT = kOffAsfRaw + 1152;            // 36 groups x 32 B max
    static constexpr int kStageBytes = ((kOffAsfT + 512 * kSfChunks) + 1023) / 1024 * 1024;
    static constexpr int kSfSlotCols = 4 + 4 * kSfChunks;         // TMEM columns per stage
};

// Kernel modes, compile-time so that each variant carries only its own code:
//   kModePlain  the layer (8x4 activation scales)
//   kModeGated  grouped GEMM1 with the SwiGLU epilogue (MoE)
//   kModeSf128  dense tiles of 128/256 tokens with 128x4 activation scales
constexpr int kModePlain = 0;
constexpr int kModeGated = 1;
constexpr int kModeSf128 = 2;

// Tokens whose split-K sum one rank owns: a multiple of 4 so partials move as
// 16-byte vectors (some ranks may own none).
__host__ __device__ constexpr int tokens_per_owner(int tt, int splits) {
    return ((tt + splits - 1) / splits + 3) & ~3;
}

// Bytes of split-K partials rank `rank` receives from its peers: one whole
// slot [128][per] FP32 from each of the other splits - 1 ranks if it owns any
// token column (columns past TT in a slot are never read), else none.
__host__ __device__ constexpr uint32_t red_bytes(int tt, int splits, int rank) {
    return rank * tokens_per_owner(tt, splits) < tt
               ? static_cast<uint32_t>((splits - 1) * 128 * 4 * tokens_per_owner(tt, splits)) : 0u;
}

struct TileInfo {
    int e, n_tile, tok0, count;
};

template <int TT>
__device__ __forceinline__ TileInfo decode_tile(int t, const GemmArgs& p, const int* prefix,
                                                const int* offs) {
    TileInfo ti;
    if (p.offsets == nullptr) {
        const int tok_tiles = (p.m + TT - 1) / TT;
        constexpr int kBand = 8;  // token tiles per band: the band's weights stay hot in L2
        const int band_size = kBand * p.n_tiles;
        const int band = t / band_size;
        const int r = t - band * band_size;
        const int g = min(kBand, tok_tiles - band * kBand);
        const int tt = band * kBand + r % g;
        ti.e = 0;
        ti.n_tile = r / g;
        ti.tok0 = tt * TT;
        ti.count = min(TT, p.m - ti.tok0);
    } else {
        int lo = 0, hi = p.experts;  // find e with prefix[e] <= t < prefix[e+1]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (prefix[mid] <= t) lo = mid; else hi = mid;
        }
        const int e = lo;
        const int seg = offs[e + 1] - offs[e];
        const int ntt = (seg + TT - 1) / TT;
        const int local = t - prefix[e];
        const int nt = local / ntt;
        const int tt = local - nt * ntt;
        ti.e = e;
        ti.n_tile = nt;
        ti.tok0 = offs[e] + tt * TT;
        ti.count = min(TT, seg - tt * TT);
    }
    return ti;
}

__device__ __forceinline__ void record_timeout(volatile uint32_t* abort_flag) {
    atomicOr(&g_gemm_error, 1u);
    *abort_flag = 1u;
}

// ----------------------------------------------------------------- kernel
// Warp roles for PIPES pipelines and E = epi_warps(TT) epilogue warps:
//   0                          producer of pipe 0      (lane 0)
//   1                          MMA issuer of pipe 0    (lane 0); TMEM alloc/free
//   2 .. 1+E                   epilogue (and fused activation quantizer)
//   2+E                        activation-scale re-order (unfused)
//   3+E .. 1+E+PIPES           producers of pipes 1..PIPES-1
//   2+E+PIPES .. E+2*PIPES     MMA issuers of pipes 1..PIPES-1
// Pipe q owns the local K blocks i with i % PIPES == q of every tile, its own
// ring of `stages` shared-memory stages and its own TMEM accumulator; the
// epilogue sums the accumulators in pipe order.
// Epilogue warps: one per TMEM lane quadrant for 32-token tiles (so that two
// CTAs with two pipelines fit one SM), two per quadrant otherwise.  16-token
// tiles take eight: the fused quantizer then gives each warp one patch (the
// decode call's quantization phase is on its critical path; measured M=16
// 5.65 -> 5.27 us, M=1 5.53 -> 4.85 us), and at 72 registers two such CTAs
// still fit an SM.
__host__ __device__ constexpr int epi_warps(int tt) { return tt == 32 ? 4 : 8; }
__host__ __device__ constexpr int num_warps(int tt, int pipes) { return 3 + epi_warps(tt) + 2 * (pipes - 1); }

struct Ctx {
    uint8_t* smem;
    uint64_t* full;
    uint64_t* empty;
    uint64_t* sfraw;
    uint64_t* acc_full;
    uint64_t* acc_empty;
    uint64_t* drain;
    volatile uint32_t* abort_flag;
    const int* prefix;
    const int* offs;
    uint32_t tmem_base;
    int stages;        // per pipe
    int tile_first, tile_stride, num_tiles, kb_begin, kb_end;
    bool fused;
};

// Jobs of pipe q in one tile of nk K blocks, and the stage/phase of a job.
template <int PIPES>
__device__ __forceinline__ int pipe_jobs(int q, int nk) {
    return q < nk ? (nk - q + PIPES - 1) / PIPES : 0;
}

template <int TT, int PIPES, int MODE>
__device__ __forceinline__ void run_producer(const GemmArgs& p, const Ctx& c, int q) {
    using G = Geometry<TT>;
    // Weights stream through once per call (a tile is read again only by the
    // token tiles right after it): first in line for eviction, so that they
    // do not push out of L2 what is read again -- the activations, which
    // every weight tile of the call reads, and what the next kernel reads
    // (GEMM1's h for GEMM2, GEMM2's output rows for the MoE finalize).
    // Measured on one box: decode 5.26 -> 5.13 us, mid 9.60 -> 9.19 us, the
    // MoE layer 125.0 -> 114.3 us, grouped gate_up 70.5 -> 66.0 us.
    const uint64_t pol_w = policy_evict_first();
    const uint64_t pol_a = policy_evict_last();
    const int nk = c.kb_end - c.kb_begin;
    const int nq = pipe_jobs<PIPES>(q, nk);
    if (nq == 0) return;
    const int S = c.stages;
    auto stage_of = [&](int jq) { return q * S + jq % S; };
    const uint32_t a_bytes = c.fused ? 0u : static_cast<uint32_t>(TT * 128);
    // 128x4 activation scales: one 512-byte tile per 128 tokens of the tile
    // that exist (the buffer holds ceil128(M) rows).
    auto sf_chunks = [&](const TileInfo& ti) {
        return MODE == kModeSf128 ? min(G::kSfChunks, (ti.count + 127) / 128) : 0;
    };
    auto issue_w = [&](const TileInfo& ti, int kb, int s) {
        uint8_t* st = c.smem + s * G::kStageBytes;
        mbar_arrive_expect_tx(&c.full[s], 16384u + 512u + a_bytes + 512u * static_cast<uint32_t>(sf_chunks(ti)));
        tma_load_2d(st + G::kOffW, &p.map_w, kb * 128, ti.e * p.n_pad + ti.n_tile * 128, &c.full[s], pol_w);
        bulk_load(st + G::kOffWsf,
                  p.wsf + ((static_cast<size_t>(ti.e) * p.n_tiles + ti.n_tile) * p.kq + kb) * 512, 512,
                  &c.full[s], pol_w);
    };
    auto issue_a = [&](const TileInfo& ti, int kb, int s) {
        uint8_t* st = c.smem + s * G::kStageBytes;
        tma_load_2d(st + G::kOffA, &p.map_a, kb * 128, ti.tok0, &c.full[s], pol_a);
        if constexpr (MODE == kModeSf128) {
            // Already in the TMEM-copy order: straight into the staging slot.
            const int nch = sf_chunks(ti);
            for (int ch = 0; ch < nch; ++ch)
                bulk_load(st + G::kOffAsfT + ch * 512,
                          p.asf128 + (static_cast<size_t>((ti.tok0 >> 7) + ch) * p.kq + kb) * 512, 512, &c.full[s],
                          pol_a);
        } else {
            mbar_arrive_expect_tx(&c.sfraw[s], static_cast<uint32_t>(p.sf_groups * 32));
            tma_load_2d(st + G::kOffAsfRaw, &p.map_asf, kb * 32, ti.tok0 >> 3, &c.sfraw[s], pol_a);
        }
    };
    // Weight bytes of the first S jobs go out before waiting for the previous
    // grid: only the activations depend on it.
    int pre = 0;
    for (int t = c.tile_first; t < c.num_tiles && pre < S; t += c.tile_stride) {
        const TileInfo ti = decode_tile<TT>(t, p, c.prefix, c.offs);
        for (int i = q; i < nk && pre < S; i += PIPES, ++pre) issue_w(ti, c.kb_begin + i, stage_of(pre));
    }
    if (!c.fused) {
        pdl_wait();
        int j = 0;
        for (int t = c.tile_first; t < c.num_tiles && j < pre; t += c.tile_stride) {
            const TileInfo ti = decode_tile<TT>(t, p, c.prefix, c.offs);
            for (int i = q; i < nk && j < pre; i += PIPES, ++j) issue_a(ti, c.kb_begin + i, stage_of(j));
        }
    }
    int jq = 0;
    bool stop = false;
    for (int t = c.tile_first; t < c.num_tiles && !stop; t += c.tile_stride) {
        const TileInfo ti = decode_tile<TT>(t, p, c.prefix, c.offs);
        for (int i = q; i < nk; i += PIPES, ++jq) {
            if (jq < pre) continue;
            const int s = stage_of(jq);
            if (!mbar_wait(&c.empty[s], ((jq / S) & 1) ^ 1, p.wait_ns)) {
                record_timeout(c.abort_flag);
                stop = true;
                break;
            }
            issue_w(ti, c.kb_begin + i, s);
            if (!c.fused) issue_a(ti, c.kb_begin + i, s);
        }
    }
    // Drain: the last use of each stage must have landed before exit.
    const int issued = jq > pre ? jq : pre;
    for (int j = issued - 1; j >= 0 && j >= issued - S; --j) {
        (void)mbar_wait(&c.full[stage_of(j)], (j / S) & 1, kDrainNs);
        if (!c.fused && MODE != kModeSf128) (void)mbar_wait(&c.sfraw[stage_of(j)], (j / S) & 1, kDrainNs);
    }
}

template <int TT, int PIPES>
__device__ __forceinline__ void run_mma(const GemmArgs& p, const Ctx& c, int q) {
    using G = Geometry<TT>;
    // Descriptors of stage 0; stage s adds s * kStageBytes (the start address
    // field is address >> 4 and never carries: shared memory < 256 KB).
    const uint64_t a_desc0 = desc_kmajor_sw128(smem_addr(c.smem + G::kOffW));
    const uint64_t b_desc0 = desc_kmajor_sw128(smem_addr(c.smem + G::kOffA));
    const uint64_t wsf_desc0 = desc_sf_32x16(smem_addr(c.smem + G::kOffWsf));
    const uint64_t asf_desc0 = desc_sf_32x16(smem_addr(c.smem + G::kOffAsfT));
    constexpr uint64_t kStageStep = static_cast<uint64_t>(G::kStageBytes >> 4);
    const int nk = c.kb_end - c.kb_begin;
    const int nq = pipe_jobs<PIPES>(q, nk);  // jobs of this pipe in one tile
    const int S = c.stages;
    const int nb = p.acc_bufs;
    int jq = 0;
    int tile_iter = 0;
    for (int t = c.tile_first; t < c.num_tiles; t += c.tile_stride, ++tile_iter) {
        const TileInfo ti = decode_tile<TT>(t, p, c.prefix, c.offs);
        const uint32_t n_mma = static_cast<uint32_t>((ti.count + 15) & ~15);
        uint32_t idesc[4];
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) idesc[kk] = idesc_mxf8(128, n_mma, kk, kk);
        // Accumulator buffer a takes tiles a, a + nb, ...: every pipe waits for
        // the epilogue to drain the buffer's previous tile, so a buffer's
        // barriers never run two phases ahead of any pipe.
        const int ab = tile_iter % nb;
        const int use = tile_iter / nb;
        const uint32_t acc = c.tmem_base + (ab * PIPES + q) * TT;
        if (use > 0 && !mbar_wait(&c.acc_empty[ab], (use - 1) & 1, p.wait_ns)) {
            record_timeout(c.abort_flag);
            break;
        }
        tc_fence_after();
        bool stop = false;
        for (int i = q; i < nk; i += PIPES, ++jq) {
            const int s = q * S + jq % S;
            if (!mbar_wait(&c.full[s], (jq / S) & 1, p.wait_ns)) {
                record_timeout(c.abort_flag);
                stop = true;
                break;
            }
            const uint64_t sd = static_cast<uint64_t>(s) * kStageStep;
            const uint32_t sfa = c.tmem_base + nb * PIPES * TT + s * G::kSfSlotCols;
            const uint32_t sfb = sfa + 4;
            tmem_copy_sf(sfa, wsf_desc0 + sd);
#pragma unroll
            for (int ch = 0; ch < G::kSfChunks; ++ch) tmem_copy_sf(sfb + 4 * ch, asf_desc0 + sd + ch * 32);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_mxf8(acc, a_desc0 + sd + 2 * kk, b_desc0 + sd + 2 * kk, idesc[kk], sfa, sfb,
                         (i > q || kk > 0) ? 1u : 0u);
            // Release the stage to its producer -- unless no later job of this
            // pipe uses it (one-tile schedules): a commit costs issue time.
            if (p.persistent || jq + S < nq) mma_commit(&c.empty[s]);
        }
        if (stop) break;
        mma_commit(&c.acc_full[ab]);  // also for a pipe with no K block in this tile
    }
    // Drain every MMA this thread issued before TMEM is released.
    mma_commit(&c.drain[q]);
    (void)mbar_wait(&c.drain[q], 0, kDrainNs);
}

template <int TT, int PIPES>
__device__ __forceinline__ void run_reorder(const GemmArgs& p, const Ctx& c, int lane) {
    using G = Geometry<TT>;
    const int nk = c.kb_end - c.kb_begin;
    const int S = c.stages;
    int tile_iter = 0;
    for (int t = c.tile_first; t < c.num_tiles; t += c.tile_stride, ++tile_iter) {
        const TileInfo ti = decode_tile<TT>(t, p, c.prefix, c.offs);
        const int off8 = ti.tok0 & 7;
        for (int i = 0; i < nk; ++i) {
            const int q = i % PIPES;
            const int jq = tile_iter * pipe_jobs<PIPES>(q, nk) + i / PIPES;
            const int s = q * S + jq % S;
            bool ok = mbar_wait(&c.sfraw[s], (jq / S) & 1, p.wait_ns);
            ok = __all_sync(0xFFFFFFFFu, ok ? 1 : 0) != 0;
            if (!ok) {
                if (lane == 0) record_timeout(c.abort_flag);
                return;
            }
            uint8_t* st = c.smem + s * G::kStageBytes;
            // Token j of the tile is word (off8 + j) of the raw 8x4 groups; the
            // TMEM-copy order puts token j of each 128-chunk at word
            // (j%32)*4 + (j%128)/32.
            const uint32_t* raw = reinterpret_cast<const uint32_t*>(st + G::kOffAsfRaw);
#pragma unroll
            for (int ch = 0; ch < G::kSfChunks; ++ch) {
                uint32_t w[4];
#pragma unroll
                for (int jq4 = 0; jq4 < 4; ++jq4) {
                    const int j = ch * 128 + jq4 * 32 + lane;
                    w[jq4] = (j < TT) ? raw[off8 + j] : 0u;
                }
                *reinterpret_cast<uint4*>(st + G::kOffAsfT + ch * 512 + lane * 16) =
                    make_uint4(w[0], w[1], w[2], w[3]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&c.full[s]);
        }
    }
}

// Fused activation quantizer (one tile per CTA).  The tile's BF16 rows are
// cut into patches of 8 token rows x one 128-wide K block; lane l of a warp
// quantizes 32-block l%4 of patch row l/4 on its own (same arithmetic as
// quant.cu), writes its 32 E4M3 bytes into the swizzled B tile and its scale
// byte into the TMEM-copy order.  Patches go round-robin over the epilogue
// warps with kBatch patches of loads in flight; after each patch the warp
// fences and arrives on the K block's full barrier, which expects one
// arrival per patch besides the producer's.
template <int TT, int PIPES>
__device__ __forceinline__ void run_fused_quant(const GemmArgs& p, const Ctx& c, int ew, int lane) {
    using G = Geometry<TT>;
    const TileInfo ti = decode_tile<TT>(c.tile_first, p, c.prefix, c.offs);
    const int nk = c.kb_end - c.kb_begin;
    // While the previous grid still runs, pull this CTA's K slice of x into
    // L2 (one bulk prefetch per token row, spread over the epilogue warps, so
    // the producer's weight loads are not delayed).  A prefetch only warms
    // L2, which every write reaches first: the loads below, issued after the
    // wait, still see what the previous grid wrote.
    for (int r = ew * 32 + lane; r < ti.count; r += epi_warps(TT) * 32)
        prefetch_l2_bulk(p.x + static_cast<size_t>(ti.tok0 + r) * p.k + c.kb_begin * 128,
                         static_cast<uint32_t>(nk) * 256u);
    pdl_wait();
    const int S = c.stages;
    constexpr int kEpi = epi_warps(TT);
    constexpr int kPatches = TT / 8;  // per K block
    constexpr int kBatch = TT == 16 ? 1 : ((PIPES == 1) ? 2 : 4);  // within the register budget
    const int total = nk * kPatches;
    const int r8 = lane >> 2;
    const int b4 = lane & 3;
    for (int p0 = ew; p0 < total; p0 += kEpi * kBatch) {
        uint4 raw[kBatch][4];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int ps = p0 + u * kEpi;
            const int i = ps / kPatches;
            const int row = (ps - i * kPatches) * 8 + r8;
#pragma unroll
            for (int v = 0; v < 4; ++v) raw[u][v] = make_uint4(0, 0, 0, 0);
            if (ps < total && row < ti.count) {
                const uint4* src = reinterpret_cast<const uint4*>(
                    p.x + static_cast<size_t>(ti.tok0 + row) * p.k + (c.kb_begin + i) * 128 + b4 * 32);
#pragma unroll
                for (int v = 0; v < 4; ++v) raw[u][v] = src[v];
            }
        }
        // The batch's loads are all in flight; each patch is then quantized
        // and published on its own, so the MMA of the first K blocks starts
        // while the later patches are still being quantized.
        uint32_t qq[kBatch][8];
        uint32_t sc[kBatch];
        auto store_patch = [&](int u, int ps) {
            const int i = ps / kPatches;
            const int row = (ps - i * kPatches) * 8 + r8;
            const int jq = i / PIPES;
            uint8_t* st = c.smem + ((i % PIPES) * S + jq % S) * G::kStageBytes;
            // Bytes [32*b4, 32*b4 + 32) of the row's 128-byte K block are
            // 16-byte chunks 2*b4 and 2*b4 + 1, swizzled with row % 8.
            uint8_t* brow = st + G::kOffA + row * 128;
            *reinterpret_cast<uint4*>(brow + (((2 * b4) ^ (row & 7)) << 4)) =
                make_uint4(qq[u][0], qq[u][1], qq[u][2], qq[u][3]);
            *reinterpret_cast<uint4*>(brow + (((2 * b4 + 1) ^ (row & 7)) << 4)) =
                make_uint4(qq[u][4], qq[u][5], qq[u][6], qq[u][7]);
            const int rr = row & 127;
            st[G::kOffAsfT + (row >> 7) * 512 + (rr & 31) * 16 + (rr >> 5) * 4 + b4] = static_cast<uint8_t>(sc[u]);
        };
        auto full_of = [&](int ps) {
            const int i = ps / kPatches;
            return &c.full[(i % PIPES) * S + (i / PIPES) % S];
        };
        // A patch whose stage is in use again must wait for the MMA to free
        // it, and that MMA may need an earlier patch of this very batch, so
        // such batches quantize everything first and then wait, store and
        // publish patch by patch.
        const bool reuse = (p0 + (kBatch - 1) * kEpi) / kPatches / PIPES >= S;
        if (!reuse) {
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                if (p0 + u * kEpi < total) {
                    sc[u] = quantize_block32(raw[u], qq[u]);
                    store_patch(u, p0 + u * kEpi);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(full_of(p0 + u * kEpi));
                }
            }
        } else {
#pragma unroll
            for (int u = 0; u < kBatch; ++u) sc[u] = quantize_block32(raw[u], qq[u]);
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int ps = p0 + u * kEpi;
                if (ps >= total) break;  // warp-uniform
                const int i = ps / kPatches;
                const int jq = i / PIPES;
                if (jq >= S) {
                    const int s = (i % PIPES) * S + jq % S;
                    bool ok = mbar_wait(&c.empty[s], ((jq / S) & 1) ^ 1, p.wait_ns);
                    ok = __all_sync(0xFFFFFFFFu, ok ? 1 : 0) != 0;
                    if (!ok) {
                        if (lane == 0) record_timeout(c.abort_flag);
                        return;
                    }
                }
                store_patch(u, ps);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(full_of(ps));
            }
        }
    }
}

// Small token tiles with one pipe keep registers low enough for two CTAs
// per SM.
template <int TT, int PIPES, int MODE>
__global__ void __launch_bounds__(32 * num_warps(TT, PIPES),
                                  ((TT <= 64 && PIPES == 1) || (TT <= 32 && PIPES == 2) || (TT == 16 && PIPES == 4)) ? 2 : 1)
    mxfp8_gemm_kernel(const __grid_constant__ GemmArgs p) {
    constexpr bool kGated = MODE == kModeGated;
    constexpr bool kSf128 = MODE == kModeSf128;
    using G = Geometry<TT>;
    constexpr int kEpi = epi_warps(TT);
    constexpr int kReorderWarp = 2 + kEpi;
    extern __shared__ uint8_t smem_dyn[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~static_cast<uintptr_t>(1023));

    // Dependent grids may launch now; they wait for this grid before reading
    // anything it writes.
    pdl_launch_dependents();

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int S = p.stages;          // per pipe
    const int ST = PIPES * S;        // all stages
    const int splits = p.splits;
    const bool reduce = splits > 1;
    const bool fused = p.x != nullptr;
    const int per = tokens_per_owner(TT, splits);

    uint8_t* partial = smem + ST * G::kStageBytes;  // split-K partials [splits][128][per] f32
    // Gated epilogue: the up half of each tile's accumulator passes through
    // xbuf [TT columns][64 rows] FP32 to the gate half.
    float* xbuf = reinterpret_cast<float*>(partial + (reduce ? splits * per * 512 : 0));
    // Gated epilogue quantizing h (p.hq): one [tokens][80 bytes] BF16 block per
    // gate-half warp, 2 x TT rows in all.
    uint8_t* hbuf = reinterpret_cast<uint8_t*>(xbuf) + (kGated ? 64 * TT * 4 : 0);
    uint8_t* ctrl = hbuf + (kGated ? 160 * TT : 0);
    Ctx c;
    c.smem = smem;
    c.full = reinterpret_cast<uint64_t*>(ctrl);
    c.empty = c.full + ST;
    c.sfraw = c.empty + ST;
    c.acc_full = c.sfraw + ST;
    c.acc_empty = c.acc_full + 2;  // acc_full[2], acc_empty[2]: one pair per accumulator buffer
    c.drain = c.acc_empty + 2;     // [PIPES]
    uint64_t* red = c.drain + PIPES;  // split-K: the peers' partials have landed
    uint64_t* xfull = red + 1;        // gated: the up half of a tile is in xbuf
    uint64_t* xempty = red + 2;       // gated: the gate half has read it
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(red + 3);
    c.abort_flag = tmem_slot + 1;
    int* prefix = reinterpret_cast<int*>(tmem_slot + 2);   // [experts + 1]
    int* offs = prefix + (kMaxExperts + 1);                 // [experts + 1]
    c.prefix = prefix;
    c.offs = offs;
    c.stages = S;
    c.fused = fused;

    // ---------------------------------------------------------------- setup
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&p.map_w);
        if (!fused) {
            tma_prefetch_desc(&p.map_a);
            if (!kSf128) tma_prefetch_desc(&p.map_asf);
        }
        for (int s = 0; s < ST; ++s) {
            // full: the producer's arrival (+ TMA bytes) and either one
            // arrival per fused-quantizer patch or the scale re-order warp's.
            mbar_init(&c.full[s], fused ? 1 + TT / 8 : (kSf128 ? 1 : 2));
            mbar_init(&c.empty[s], 1);
            mbar_init(&c.sfraw[s], 1);
        }
        for (int ab = 0; ab < 2; ++ab) {
            mbar_init(&c.acc_full[ab], PIPES);
            mbar_init(&c.acc_empty[ab], kEpi);
        }
        for (int q = 0; q < PIPES; ++q) mbar_init(&c.drain[q], 1);
        if (kGated) {
            mbar_init(xfull, kEpi / 2);   // one arrival per up-half warp
            mbar_init(xempty, kEpi / 2);  // one arrival per gate-half warp
        }
        if (reduce) {
            // Bytes the other ranks push into this rank's slice of the tile.
            mbar_init(red, 1);
            mbar_arrive_expect_tx(red, red_bytes(TT, splits, static_cast<int>(cluster_rank())));
        }
        *c.abort_flag = 0u;
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc(tmem_slot, p.tmem_cols);
    if (warp == 2 && p.offsets != nullptr) {
        // Grouped: per-expert tile counts -> exclusive prefix (tiles ordered
        // expert-major, then n-tile, then token tile).  The offsets were
        // written before this layer's first kernel began.
        const int ne = p.experts;
        int carry = 0;
        for (int base = 0; base <= ne; base += 32) {
            const int i = base + lane;
            int o = (i <= ne) ? p.offsets[i] : 0;
            if (i <= ne) offs[i] = o;
            int o_next = __shfl_down_sync(0xFFFFFFFFu, o, 1);
            if (lane == 31) o_next = (i + 1 <= ne) ? p.offsets[i + 1] : 0;
            int cnt = 0;
            if (i < ne) {
                const int seg = o_next - o;
                cnt = seg > 0 ? p.n_tiles * ((seg + TT - 1) / TT) : 0;
            }
            int incl = cnt;  // inclusive warp scan
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int v = __shfl_up_sync(0xFFFFFFFFu, incl, d);
                if (lane >= d) incl += v;
            }
            if (i <= ne) prefix[i] = carry + incl - cnt;
            carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    c.tmem_base = *tmem_slot;
    // Split-K lifetime protocol (cluster barrier, two phases, every thread):
    // phase 1 (arrive here, wait before the first remote store) guarantees
    // that every peer has initialised its barriers; phase 2 (arrive once this
    // thread's pushes are issued, wait before exit) keeps every CTA alive
    // until no peer can push into its shared memory any more.
    if (reduce) cluster_arrive_relaxed();

    // Work assignment: a list of (tile, K range).
    int rank = 0;
    if (!p.persistent) {
        rank = reduce ? static_cast<int>(cluster_rank()) : 0;
        c.tile_first = reduce ? static_cast<int>(cluster_id_x()) : static_cast<int>(blockIdx.x);
        c.tile_stride = 1 << 30;
        c.num_tiles = c.tile_first + 1;
        c.kb_begin = (rank * p.kq) / splits;
        c.kb_end = ((rank + 1) * p.kq) / splits;
    } else {
        c.tile_first = blockIdx.x;
        c.tile_stride = gridDim.x;
        c.num_tiles = (p.offsets == nullptr) ? p.num_tiles : prefix[p.experts];
        c.kb_begin = 0;
        c.kb_end = p.kq;
    }
    const int nk = c.kb_end - c.kb_begin;

    if (warp == 0 || (warp > kReorderWarp && warp < kReorderWarp + PIPES)) {
        if (lane == 0) run_producer<TT, PIPES, MODE>(p, c, warp == 0 ? 0 : warp - kReorderWarp);
        __syncwarp();
    } else if (warp == 1 || (warp >= kReorderWarp + PIPES && warp < num_warps(TT, PIPES))) {
        if (lane == 0) run_mma<TT, PIPES>(p, c, warp == 1 ? 0 : warp - (kReorderWarp + PIPES) + 1);
        __syncwarp();
    } else if (warp == kReorderWarp) {
        if (!fused && !kSf128) run_reorder<TT, PIPES>(p, c, lane);
        __syncwarp();
    } else {
        const int ew = warp - 2;  // warps 2 .. 1+kEpi
        if (fused) run_fused_quant<TT, PIPES>(p, c, ew, lane);
        if (reduce) {
            __syncwarp();
            cluster_wait();  // phase 1: peers are running (latency hidden behind the MMAs)
        }
        // ------------------------------------------------------- epilogue
        const int quad = warp & 3;             // TMEM lanes [32*quad, 32*quad + 32)
        const int half = ew >> 2;              // token columns [half*kCols, (half+1)*kCols)
        constexpr int kCols = TT * 4 / kEpi;
        const int col0 = half * kCols;
        const int n_active = nk < PIPES ? nk : PIPES;
        const int nl = quad * 32 + lane;       // weight row within the tile
        float acc[kCols];
        float b = 0.0f;
        int tile_iter = 0;
        for (int t = c.tile_first; t < c.num_tiles; t += c.tile_stride, ++tile_iter) {
            const TileInfo ti = decode_tile<TT>(t, p, prefix, offs);
            const int n = ti.n_tile * 128 + nl;
            b = (p.bias && n < p.n) ? __bfloat162float(p.bias[static_cast<size_t>(ti.e) * p.n + n]) : 0.0f;
            const int ab = tile_iter % p.acc_bufs;
            bool ok = mbar_wait(&c.acc_full[ab], (tile_iter / p.acc_bufs) & 1, p.wait_ns);
            ok = __all_sync(0xFFFFFFFFu, ok ? 1 : 0) != 0;
            if (!ok) { if (lane == 0) record_timeout(c.abort_flag); break; }
            tc_fence_after();
#pragma unroll
            for (int i = 0; i < kCols; ++i) acc[i] = 0.0f;
            for (int q = 0; q < n_active; ++q) {  // pipe order: deterministic sums
                const uint32_t taddr =
                    c.tmem_base + (ab * PIPES + q) * TT + (static_cast<uint32_t>(quad * 32) << 16) + col0;
                uint32_t r[kCols];
                if constexpr (kCols >= 32) {
#pragma unroll
                    for (int cc = 0; cc < kCols / 32; ++cc) {
                        uint32_t r32[32];
                        tmem_load_32(taddr + cc * 32, r32);
#pragma unroll
                        for (int i = 0; i < 32; ++i) r[cc * 32 + i] = r32[i];
                    }
                } else if constexpr (kCols == 16) {
                    tmem_load_16(taddr, r);
                } else {
                    tmem_load_8(taddr, r);
                }
                tmem_load_wait();
#pragma unroll
                for (int i = 0; i < kCols; ++i) acc[i] += __uint_as_float(r[i]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&c.acc_empty[ab]);

            if (reduce) {
                // Stage the partial tile in the idle pipeline stages (every MMA
                // has completed) as 4-column chunks: staging[col/4][row][col%4].
                // Rank o's slice, columns [o*per, o*per + per), is then one
                // contiguous run of per * 512 bytes.
                float4* stg = reinterpret_cast<float4*>(smem);
#pragma unroll
                for (int j = 0; j < kCols; j += 4)
                    stg[((col0 + j) >> 2) * 128 + nl] = make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
                fence_proxy_async_smem();
            } else if constexpr (kGated) {
                // SwiGLU: rows [0, 64) of the tile are gate rows, [64, 128) the
                // matching up rows (gated-row order of the prepared weights);
                // output feature ti.n_tile * 64 + nl of h = silu(gate) * up.
                const bool up_half = nl >= 64;  // warp-uniform
                const int inter = p.n >> 1;
                if (up_half) {
                    bool okx = tile_iter == 0 || mbar_wait(xempty, (tile_iter - 1) & 1, p.wait_ns);
                    okx = __all_sync(0xFFFFFFFFu, okx ? 1 : 0) != 0;
                    if (!okx) { if (lane == 0) record_timeout(c.abort_flag); break; }
#pragma unroll
                    for (int j = 0; j < kCols; ++j) xbuf[(col0 + j) * 64 + (nl - 64)] = acc[j];
                    __syncwarp();
                    if (lane == 0) mbar_arrive(xfull);
                } else {
                    bool okx = mbar_wait(xfull, tile_iter & 1, p.wait_ns);
                    okx = __all_sync(0xFFFFFFFFu, okx ? 1 : 0) != 0;
                    if (!okx) { if (lane == 0) record_timeout(c.abort_flag); break; }
                    const int f = ti.n_tile * 64 + nl;
                    const int jmax = min(kCols, ti.count - col0);
                    if (p.hq != nullptr) {
                        // h goes straight to MXFP8 for the next GEMM, exactly as
                        // the activation quantizer turns the BF16 h: this warp's
                        // 32 features (one K block of h, f/32) x its tokens are
                        // written to its shared-memory block as BF16, one
                        // 80-byte row per token (16-byte reads of different rows
                        // then hit different banks), and lane l quantizes token
                        // row l with quant_block.cuh's routine: two 16-byte
                        // stores of E4M3 bytes and one scale byte (8x4 layout).
                        uint8_t* tp = hbuf + ((quad & 1) + 2 * half) * (kCols * 80);
#pragma unroll
                        for (int j = 0; j < kCols; ++j) {
                            const float g = acc[j];
                            const float hv = g / (1.0f + expf(-g)) * xbuf[(col0 + j) * 64 + nl];
                            *reinterpret_cast<unsigned short*>(tp + j * 80 + lane * 2) =
                                __bfloat16_as_ushort(__float2bfloat16_rn(hv));
                        }
                        __syncwarp();
                        const int kb = inter >> 5;
                        const int fb = f - lane;  // first feature of the block
                        const int b = fb >> 5;
                        for (int jj = lane; jj < jmax; jj += 32) {
                            const uint4* src = reinterpret_cast<const uint4*>(tp + jj * 80);
                            const uint4 raw[4] = {src[0], src[1], src[2], src[3]};
                            uint32_t qq[8];
                            const uint32_t sc = quantize_block32(raw, qq);
                            const int64_t row = ti.tok0 + col0 + jj;
                            if (store_ok(row * inter + fb, 32, static_cast<int64_t>(p.m) * inter)) {
                                uint4* dst = reinterpret_cast<uint4*>(p.hq + row * inter + fb);
                                dst[0] = make_uint4(qq[0], qq[1], qq[2], qq[3]);
                                dst[1] = make_uint4(qq[4], qq[5], qq[6], qq[7]);
                            }
                            const int64_t o = ((row >> 3) * (kb >> 2) + (b >> 2)) * 32 + (row & 7) * 4 + (b & 3);
                            if (store_ok(o, 1, ((static_cast<int64_t>(p.m) + 7) >> 3) * 8 * kb))
                                p.hsf[o] = static_cast<uint8_t>(sc);
                        }
                        __syncwarp();  // the block is rewritten for the next tile
                    } else {
                        __nv_bfloat16* hp = p.y + static_cast<size_t>(ti.tok0 + col0) * inter + f;
#pragma unroll
                        for (int j = 0; j < kCols; ++j) {
                            const float g = acc[j];
                            const float hv = g / (1.0f + expf(-g)) * xbuf[(col0 + j) * 64 + nl];
                            if (j < jmax && store_ok(static_cast<int64_t>(ti.tok0 + col0 + j) * inter + f, 1,
                                                     static_cast<int64_t>(p.m) * inter))
                                hp[static_cast<size_t>(j) * inter] = __float2bfloat16_rn(hv);
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(xempty);
                }
            } else if (n < p.n) {
                const int jmax = min(kCols, ti.count - col0);
                __nv_bfloat16* yp = p.y + static_cast<size_t>(ti.tok0 + col0) * p.n + n;
#pragma unroll
                for (int j = 0; j < kCols; ++j)
                    if (j < jmax && store_ok(static_cast<int64_t>(ti.tok0 + col0 + j) * p.n + n, 1,
                                             static_cast<int64_t>(p.m) * p.n))
                        yp[static_cast<size_t>(j) * p.n] = __float2bfloat16_rn(acc[j] + b);
            }
        }
        if (reduce) {
            // Push: once every epilogue warp has staged its partials, one
            // thread hands each peer its slice (one bulk copy per peer into
            // the peer's slot [rank], counted on the peer's `red` barrier).
            // Nothing is pushed if any role of this CTA gave up.
            named_barrier_sync(1, kEpi * 32);
            const bool push = *c.abort_flag == 0u;
            const uint32_t slot_bytes = static_cast<uint32_t>(per * 512);
            if (push && ew == 0 && lane < splits && lane != rank && red_bytes(TT, splits, lane) > 0) {
                // Lane o of the first epilogue warp issues the copy to peer o.
                bulk_copy_to_peer(map_to_rank(smem_addr(partial) + rank * slot_bytes, static_cast<uint32_t>(lane)),
                                  smem + lane * slot_bytes, slot_bytes,
                                  map_to_rank(smem_addr(red), static_cast<uint32_t>(lane)));
            }
            // Owner: columns [rank*per, rank*per + per) of the tile, spread
            // over all epilogue threads (row et % 128, every (kEpi/4)-th
            // 4-column chunk), summed over the ranks in rank order.
            const bool owns = red_bytes(TT, splits, rank) > 0;
            const int et = ew * 32 + lane;
            const int rn = et & 127;
            const TileInfo ti = decode_tile<TT>(c.tile_first, p, prefix, offs);
            const int n = ti.n_tile * 128 + rn;
            const float bn = (owns && p.bias && n < p.n)
                                 ? __bfloat162float(p.bias[static_cast<size_t>(ti.e) * p.n + n]) : 0.0f;
            bool landed = !owns;
            if (owns) {
                landed = push && mbar_wait(red, 0, p.wait_ns);
                landed = __all_sync(0xFFFFFFFFu, landed ? 1 : 0) != 0;
                if (!landed) {
                    if (push && lane == 0) record_timeout(c.abort_flag);
                    // Error path: let copies already in flight land (their
                    // sources stay alive until phase 2 completes).
                    (void)mbar_wait(red, 0, kDrainNs);
                }
            }
            // Phase 2: every copy into this CTA has landed (or the drain ran
            // out), so the copies that read the peers' staging areas are done.
            __syncwarp();
            cluster_arrive_relaxed();
            if (owns && landed && push && n < p.n) {
                const float4* own = reinterpret_cast<const float4*>(smem) + rank * (per / 4) * 128;
                const float4* part = reinterpret_cast<const float4*>(partial);
                const int o0 = rank * per;
                const int cmax = min(per, ti.count - o0);
                for (int q = et >> 7; q * 4 < cmax; q += kEpi / 4) {
                    float4 sum = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                    for (int r = 0; r < splits; ++r) {
                        const float4 v = (r == rank ? own : part + r * (per / 4) * 128)[q * 128 + rn];
                        sum.x += v.x; sum.y += v.y; sum.z += v.z; sum.w += v.w;
                    }
                    const float sv[4] = {sum.x, sum.y, sum.z, sum.w};
                    __nv_bfloat16* yq = p.y + static_cast<size_t>(ti.tok0 + o0 + q * 4) * p.n + n;
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        if (q * 4 + i < cmax &&
                            store_ok(static_cast<int64_t>(ti.tok0 + o0 + q * 4 + i) * p.n + n, 1,
                                     static_cast<int64_t>(p.m) * p.n))
                            yq[static_cast<size_t>(i) * p.n] = __float2bfloat16_rn(sv[i] + bn);
                }
            }
        }
        __syncwarp();
    }

    if (reduce) {
        __syncwarp();
        const bool epi = warp >= 2 && warp < 2 + kEpi;
        if (!epi) {
            cluster_wait();            // phase 1
            cluster_arrive_relaxed();  // phase 2: this warp receives nothing
        }
        cluster_wait();  // phase 2: every owner has received all of its slice
    }

    // -------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(c.tmem_base, p.tmem_cols);
    }
}

// ------------------------------------------------------- dual-tile kernel
// Large-M dense schedule.  A CTA tile is two adjacent 128-row weight tiles
// (256 output features) x TT tokens (TT = 144, 160, 176 or 192; a multiple
// of 16, the MMA's N step, and of 8, the activation scale groups).  The token tile and its scales are loaded
// once per K block and serve both weight tiles; one MMA-issuing thread per
// weight tile runs over all K blocks into its own TMEM accumulator.  Both
// issuers feed the same tensor core, so together they keep it busy although
// each pays a fixed cost per tcgen05 instruction.
//   warp 0       producer (lane 0): both weight tiles, both scale tiles, the
//                token tile, the raw 8x4 token scales
//   warps 1, 11  MMA issuers of weight tile 0 / 1 (lane 0); warp 1 owns TMEM
//   warps 2..9   epilogue: warp 2+e serves accumulator e/4, lane quadrant
//                warp%4, 32 token columns at a time, stored from registers
//   warp 10      token-scale re-order into the TMEM-copy order
template <int TT, bool SF128 = false>
struct DualGeometry {
    static constexpr int kSfChunks = (TT + 127) / 128;
    static constexpr int kOffW0 = 0;
    static constexpr int kOffW1 = 16384;
    static constexpr int kOffA = 32768;
    static constexpr int kOffWsf0 = kOffA + TT * 128;
    static constexpr int kOffWsf1 = kOffWsf0 + 512;
    // The raw 8x4 token-scale groups land in the area that then holds them in
    // the TMEM-copy order: the re-order warp reads all its words before it
    // writes (in place).  Sharing the area is what lets 176-token tiles run
    // four 56 KB stages.
    static constexpr int kOffAsfT = kOffWsf1 + 512;
    static constexpr int kOffAsfRaw = kOffAsfT;
    // With 128x4 token scales (SF128) the raw area holds the 512-byte scale
    // tiles of every 128-row tile the token tile touches: up to three.
    static constexpr int kRawTiles = SF128 ? (TT + 126) / 128 + 1 : 0;
    static constexpr int kAreaBytes = SF128 && 512 * kRawTiles > 512 * kSfChunks ? 512 * kRawTiles : 512 * kSfChunks;
    static constexpr int kStageBytes = ((kOffAsfT + kAreaBytes) + 1023) / 1024 * 1024;
    static constexpr int kSlotCols = 4 + 4 * kSfChunks;  // per pipe per stage
    static_assert(SF128 || (TT / 8 + 1) * 32 <= 512 * kSfChunks, "raw scale groups must fit the shared area");
};

constexpr int kDualThreads = 12 * 32;

// Dense tiles over (weight-tile pair, token tile), token tiles banded by 8 so
// a band's weights stay in L2.
template <int TT>
__device__ __forceinline__ TileInfo decode_dual(int t, const GemmArgs& p) {
    const int pairs = (p.n_tiles + 1) >> 1;
    const int tok_tiles = (p.m + TT - 1) / TT;
    constexpr int kBand = 8;
    const int band_size = kBand * pairs;
    const int band = t / band_size;
    const int r = t - band * band_size;
    const int g = min(kBand, tok_tiles - band * kBand);
    const int tt = band * kBand + r % g;
    TileInfo ti;
    ti.e = 0;
    ti.n_tile = 2 * (r / g);  // first of the pair
    ti.tok0 = tt * TT;
    ti.count = min(TT, p.m - ti.tok0);
    return ti;
}

// 128x4 scale tiles (of 128 rows) a token tile starting at tok0 touches,
// counting none past the last row tile of an m-row buffer (ceil128(m) rows).
template <int TT>
__host__ __device__ __forceinline__ int dual_raw_tiles(int tok0, int m) {
    const int last = (m + 127) / 128 - 1;
    const int r1 = (tok0 + TT - 1) >> 7;
    return (r1 < last ? r1 : last) - (tok0 >> 7) + 1;
}

template <int TT, bool SF128 = false>
__global__ void __launch_bounds__(kDualThreads, 1) mxfp8_gemm_dual_kernel(const __grid_constant__ GemmArgs p) {
    using G = DualGeometry<TT, SF128>;
    extern __shared__ uint8_t smem_dyn[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~static_cast<uintptr_t>(1023));
    pdl_launch_dependents();

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int S = p.stages;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * G::kStageBytes);
    uint64_t* empty = full + S;
    uint64_t* sfraw = empty + S;
    uint64_t* acc_full = sfraw + S;   // [2], one per accumulator
    uint64_t* acc_empty = acc_full + 2;  // [2]
    uint64_t* drain = acc_empty + 2;  // [2]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 2);
    volatile uint32_t* abort_flag = tmem_slot + 1;

    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&p.map_w);
        tma_prefetch_desc(&p.map_a);
        tma_prefetch_desc(&p.map_asf);
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 2);   // producer (+ bytes), re-order warp
            mbar_init(&empty[s], 2);  // both MMA issuers
            mbar_init(&sfraw[s], 1);
        }
        for (int q = 0; q < 2; ++q) {
            mbar_init(&acc_full[q], 1);   // its MMA issuer
            mbar_init(&acc_empty[q], 4);  // its four epilogue warps
        }
        mbar_init(&drain[0], 1);
        mbar_init(&drain[1], 1);
        *abort_flag = 0u;
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc(tmem_slot, p.tmem_cols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int tile_first = blockIdx.x;
    const int tile_stride = gridDim.x;
    const int num_tiles = p.num_tiles;
    const int nk = p.kq;

    if (warp == 0) {
        // ------------------------------------------------------- producer
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_normal();
            const uint64_t pol_a = policy_evict_last();
            auto issue_w = [&](const TileInfo& ti, int kb, int s) {
                uint8_t* st = smem + s * G::kStageBytes;
                const bool has1 = ti.n_tile + 1 < p.n_tiles;
                mbar_arrive_expect_tx(&full[s], 2u * 16384u + (has1 ? 1024u : 512u) +
                                                    static_cast<uint32_t>(TT * 128));
                tma_load_2d(st + G::kOffW0, &p.map_w, kb * 128, ti.n_tile * 128, &full[s], pol_w);
                tma_load_2d(st + G::kOffW1, &p.map_w, kb * 128, (ti.n_tile + 1) * 128, &full[s], pol_w);
                bulk_load(st + G::kOffWsf0, p.wsf + (static_cast<size_t>(ti.n_tile) * p.kq + kb) * 512, 512,
                          &full[s], pol_w);
                if (has1)
                    bulk_load(st + G::kOffWsf1, p.wsf + (static_cast<size_t>(ti.n_tile + 1) * p.kq + kb) * 512,
                              512, &full[s], pol_w);
            };
            auto issue_a = [&](const TileInfo& ti, int kb, int s) {
                uint8_t* st = smem + s * G::kStageBytes;
                tma_load_2d(st + G::kOffA, &p.map_a, kb * 128, ti.tok0, &full[s], pol_a);
                if constexpr (SF128) {
                    // One box: the 512-byte 128x4 scale tiles (K block kb)
                    // of kRawTiles row tiles from the token tile's first;
                    // rows past the buffer's last tile read as zero.
                    mbar_arrive_expect_tx(&sfraw[s], static_cast<uint32_t>(G::kRawTiles * 512));
                    tma_load_2d(st + G::kOffAsfRaw, &p.map_asf, kb * 128, ti.tok0 >> 7, &sfraw[s], pol_a);
                } else {
                    mbar_arrive_expect_tx(&sfraw[s], static_cast<uint32_t>(p.sf_groups * 32));
                    tma_load_2d(st + G::kOffAsfRaw, &p.map_asf, kb * 32, ti.tok0 >> 3, &sfraw[s], pol_a);
                }
            };
            int pre = 0;
            for (int t = tile_first; t < num_tiles && pre < S; t += tile_stride) {
                const TileInfo ti = decode_dual<TT>(t, p);
                for (int kb = 0; kb < nk && pre < S; ++kb, ++pre) issue_w(ti, kb, pre);
            }
            pdl_wait();
            {
                int j = 0;
                for (int t = tile_first; t < num_tiles && j < pre; t += tile_stride) {
                    const TileInfo ti = decode_dual<TT>(t, p);
                    for (int kb = 0; kb < nk && j < pre; ++kb, ++j) issue_a(ti, kb, j);
                }
            }
            int job = 0;
            bool stop = false;
            for (int t = tile_first; t < num_tiles && !stop; t += tile_stride) {
                const TileInfo ti = decode_dual<TT>(t, p);
                for (int kb = 0; kb < nk; ++kb, ++job) {
                    if (job < pre) continue;
                    const int s = job % S;
                    if (!mbar_wait(&empty[s], ((job / S) & 1) ^ 1, p.wait_ns)) {
                        record_timeout(abort_flag);
                        stop = true;
                        break;
                    }
                    issue_w(ti, kb, s);
                    issue_a(ti, kb, s);
                }
            }
            const int issued = job > pre ? job : pre;
            for (int j = issued - 1; j >= 0 && j >= issued - S; --j) {
                (void)mbar_wait(&full[j % S], (j / S) & 1, kDrainNs);
                (void)mbar_wait(&sfraw[j % S], (j / S) & 1, kDrainNs);
            }
        }
        __syncwarp();
    } else if (warp == 1 || warp == 11) {
        // ------------------------------------------------------- MMA issuers
        if (lane == 0) {
            const int q = warp == 1 ? 0 : 1;
            const uint64_t a_desc0 = desc_kmajor_sw128(smem_addr(smem + (q ? G::kOffW1 : G::kOffW0)));
            const uint64_t b_desc0 = desc_kmajor_sw128(smem_addr(smem + G::kOffA));
            const uint64_t wsf_desc0 = desc_sf_32x16(smem_addr(smem + (q ? G::kOffWsf1 : G::kOffWsf0)));
            const uint64_t asf_desc0 = desc_sf_32x16(smem_addr(smem + G::kOffAsfT));
            constexpr uint64_t kStageStep = static_cast<uint64_t>(G::kStageBytes >> 4);
            const uint32_t acc = tmem_base + q * TT;
            int s = 0;
            uint32_t phase = 0;
            int tile_iter = 0;
            for (int t = tile_first; t < num_tiles; t += tile_stride, ++tile_iter) {
                const TileInfo ti = decode_dual<TT>(t, p);
                const uint32_t n_mma = static_cast<uint32_t>((ti.count + 15) & ~15);
                uint32_t idesc[4];
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) idesc[kk] = idesc_mxf8(128, n_mma, kk, kk);
                if (tile_iter > 0 && !mbar_wait(&acc_empty[q], (tile_iter - 1) & 1, p.wait_ns)) {
                    record_timeout(abort_flag);
                    break;
                }
                tc_fence_after();
                bool stop = false;
                for (int kb = 0; kb < nk; ++kb) {
                    if (!mbar_wait(&full[s], phase, p.wait_ns)) {
                        record_timeout(abort_flag);
                        stop = true;
                        break;
                    }
                    const uint64_t sd = static_cast<uint64_t>(s) * kStageStep;
                    const uint32_t sfa = tmem_base + 2 * TT + (s * 2 + q) * G::kSlotCols;
                    const uint32_t sfb = sfa + 4;
                    tmem_copy_sf(sfa, wsf_desc0 + sd);
#pragma unroll
                    for (int ch = 0; ch < G::kSfChunks; ++ch) tmem_copy_sf(sfb + 4 * ch, asf_desc0 + sd + ch * 32);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_mxf8(acc, a_desc0 + sd + 2 * kk, b_desc0 + sd + 2 * kk, idesc[kk], sfa, sfb,
                                 (kb > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(&empty[s]);
                    if (++s == S) { s = 0; phase ^= 1u; }
                }
                if (stop) break;
                mma_commit(&acc_full[q]);
            }
            mma_commit(&drain[q]);
            (void)mbar_wait(&drain[q], 0, kDrainNs);
        }
        __syncwarp();
    } else if (warp == 10) {
        // ------------------------------------------- token-scale re-order
        int job = 0;
        bool stop = false;
        for (int t = tile_first; t < num_tiles && !stop; t += tile_stride) {
            const TileInfo ti = decode_dual<TT>(t, p);
            const int off8 = ti.tok0 & 7;
            const int r0 = ti.tok0 >> 7;
            const int nt = SF128 ? dual_raw_tiles<TT>(ti.tok0, p.m) : 0;
            for (int kb = 0; kb < nk; ++kb, ++job) {
                const int s = job % S;
                bool ok = mbar_wait(&sfraw[s], (job / S) & 1, p.wait_ns);
                ok = __all_sync(0xFFFFFFFFu, ok ? 1 : 0) != 0;
                if (!ok) {
                    if (lane == 0) record_timeout(abort_flag);
                    stop = true;
                    break;
                }
                uint8_t* st = smem + s * G::kStageBytes;
                const uint32_t* raw = reinterpret_cast<const uint32_t*>(st + G::kOffAsfRaw);
                // In place: every word is read before any is written.
                uint32_t w[G::kSfChunks][4];
#pragma unroll
                for (int ch = 0; ch < G::kSfChunks; ++ch)
#pragma unroll
                    for (int jq = 0; jq < 4; ++jq) {
                        const int j = ch * 128 + jq * 32 + lane;
                        if constexpr (SF128) {
                            // Row g's word (its four block scales) sits at
                            // (g % 32) * 4 + (g % 128) / 32 of its row tile.
                            const int g = ti.tok0 + j;
                            const int rt = (g >> 7) - r0;
                            w[ch][jq] = (j < TT && rt < nt) ? raw[rt * 128 + (g & 31) * 4 + ((g & 127) >> 5)] : 0u;
                        } else {
                            w[ch][jq] = (j < TT) ? raw[off8 + j] : 0u;
                        }
                    }
                __syncwarp();
#pragma unroll
                for (int ch = 0; ch < G::kSfChunks; ++ch)
                    *reinterpret_cast<uint4*>(st + G::kOffAsfT + ch * 512 + lane * 16) =
                        make_uint4(w[ch][0], w[ch][1], w[ch][2], w[ch][3]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&full[s]);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------- epilogue
        // The warp's whole accumulator slice (its 32 output features x the
        // tile's columns) is read from TMEM 32 columns at a time, biased and
        // rounded to BF16 into registers (two columns per register), and only
        // then is the accumulator released: the issuer's next tile waits for
        // the TMEM reads alone, not for the stores.  Stores straight from
        // registers: lane l holds output feature n0 + l, so each store
        // instruction of the warp writes one token's 64-byte row segment.
        // (No shared staging: the 16 KB it would take buys a fourth pipeline
        // stage for tiles of <= 160 tokens.)
        const int ew = warp - 2;
        const int q = ew >> 2;   // accumulator / weight tile of the pair
        const int quad = warp & 3;
        int tile_iter = 0;
        for (int t = tile_first; t < num_tiles; t += tile_stride, ++tile_iter) {
            const TileInfo ti = decode_dual<TT>(t, p);
            const int n0 = (ti.n_tile + q) * 128 + quad * 32;  // this warp's 32 output features
            const int n = n0 + lane;
            const float b = (p.bias && n < p.n) ? __bfloat162float(p.bias[n]) : 0.0f;
            bool ok = mbar_wait(&acc_full[q], tile_iter & 1, p.wait_ns);
            ok = __all_sync(0xFFFFFFFFu, ok ? 1 : 0) != 0;
            if (!ok) { if (lane == 0) record_timeout(abort_flag); break; }
            tc_fence_after();
            const uint32_t taddr = tmem_base + q * TT + (static_cast<uint32_t>(quad * 32) << 16);
            uint32_t hv[TT / 2];  // BF16 pairs: columns 2i, 2i + 1 of the slice
            // 16 columns per TMEM load (TT is a multiple of 16: no load
            // reaches past this accumulator's own columns).
#pragma unroll
            for (int h = 0; h < TT / 16; ++h) {
                uint32_t r[16];
                tmem_load_16(taddr + h * 16, r);
                tmem_load_wait();
#pragma unroll
                for (int i = 0; i < 16; i += 2) {
                    const __nv_bfloat162 v2 = __floats2bfloat162_rn(__uint_as_float(r[i]) + b,
                                                                    __uint_as_float(r[i + 1]) + b);
                    hv[h * 8 + i / 2] = *reinterpret_cast<const uint32_t*>(&v2);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[q]);  // accumulator read: the issuer may go on
            if (n0 < p.n && n < p.n) {
                // One pointer walks the tile's token rows.
                __nv_bfloat16* yp = p.y + static_cast<size_t>(ti.tok0) * p.n + n;
                const size_t row = static_cast<size_t>(p.n);
                const int cnt = ti.count;
#pragma unroll
                for (int k = 0; k < TT / 2; ++k) {
                    const uint32_t w2 = hv[k];
                    if (2 * k < cnt && store_ok(static_cast<int64_t>(ti.tok0 + 2 * k) * p.n + n, 1,
                                                static_cast<int64_t>(p.m) * p.n))
                        *yp = __ushort_as_bfloat16(static_cast<unsigned short>(w2 & 0xFFFFu));
                    yp += row;
                    if (2 * k + 1 < cnt && store_ok(static_cast<int64_t>(ti.tok0 + 2 * k + 1) * p.n + n, 1,
                                                    static_cast<int64_t>(p.m) * p.n))
                        *yp = __ushort_as_bfloat16(static_cast<unsigned short>(w2 >> 16));
                    yp += row;
                }
            }
            __syncwarp();
        }
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, p.tmem_cols);
    }
}

// ------------------------------------------------------------------- host
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = []() -> EncodeTiledFn {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<EncodeTiledFn>(ptr);
    }();
    return fn;
}

bool encode_2d(CUtensorMap* map, const void* base, CUtensorMapDataType type, uint64_t inner, uint64_t outer,
               uint64_t row_stride, uint32_t box_inner, uint32_t box_outer, bool swizzle128) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_stride};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, type, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_2d_u8(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                  uint64_t row_stride, uint32_t box_inner, uint32_t box_outer, bool swizzle128) {
    return encode_2d(map, base, CU_TENSOR_MAP_DATA_TYPE_UINT8, inner, outer, row_stride, box_inner, box_outer,
                     swizzle128);
}

uint32_t pow2_cols(int need) {
    uint32_t c = 32;
    while (c < static_cast<uint32_t>(need)) c <<= 1;
    return c;
}

struct LaunchPlan {
    int stages;  // per pipe
    uint32_t tmem_cols;
    size_t smem;
    int partial;
};

template <int TT, int PIPES>
LaunchPlan plan_for(int splits, bool persistent, int kq, bool gated) {
    using G = Geometry<TT>;
    LaunchPlan lp;
    // Pipeline depth: as many stages as fit next to the partial buffer and
    // control block, at most 8 in all, split evenly between the pipes (a
    // one-tile CTA never needs more than its K blocks).
    const int ctrl = 8 * 64 + 8 + 4 * 2 * (kMaxExperts + 1) + 64;  // barriers, slots, prefix/offsets
    lp.partial = splits > 1 ? splits * tokens_per_owner(TT, splits) * 512 : 0;
    const int xbuf = gated ? 64 * TT * 4 + 160 * TT : 0;  // up-half exchange + h quantization blocks
    const int budget = 227 * 1024 - 1024 - ctrl - lp.partial - xbuf;
    int stages = budget / (PIPES * G::kStageBytes);
    if (stages * PIPES > 8) stages = 8 / PIPES;
    if (!persistent) {
        const int nk = (kq + splits - 1) / splits;
        const int nq = (nk + PIPES - 1) / PIPES;
        if (stages > nq) stages = nq;
    }
    if (splits > 1) {
        // The split-K partials are staged in the pipeline stages: keep room
        // for one [128][per] FP32 slot per rank.
        const int staging = splits * 128 * tokens_per_owner(TT, splits) * 4;
        const int need = (staging + PIPES * G::kStageBytes - 1) / (PIPES * G::kStageBytes);
        if (stages < need) stages = need;
    }
    lp.stages = stages;
    lp.tmem_cols = pow2_cols(PIPES * TT + PIPES * stages * G::kSfSlotCols);
    lp.smem = 1024 + static_cast<size_t>(PIPES * stages) * G::kStageBytes + lp.partial + xbuf + ctrl;
    return lp;
}

template <int TT, int PIPES, int MODE>
cudaError_t launch_tt(const GemmProblem& pr, const GemmSchedule& sch, int num_sms, cudaStream_t s,
                      bool* encode_failed) {
    constexpr int kThreads = 32 * num_warps(TT, PIPES);
    using G = Geometry<TT>;
    GemmArgs a;
    memset(&a, 0, sizeof(a));
    const int64_t m8 = (pr.m + 7) / 8 * 8;
    const bool fused = sch.fuse_quant && pr.x != nullptr;
    // One TMA box per token tile: the producer is a single thread and every
    // TMA instruction costs issue time.  Rows past M are zero-filled; rows past
    // a grouped segment belong to the next expert and are never stored.
    a.box_rows = TT;
    a.sf_groups = TT / 8 + 1;
    bool ok = encode_2d_u8(&a.map_w, pr.wq, pr.k, pr.experts * pr.n_pad, pr.k, 128, 128, true);
    if (ok && !fused)
        ok = encode_2d_u8(&a.map_a, pr.qa, pr.k, pr.m, pr.k, 128, a.box_rows, true) &&
             (pr.sf128 || encode_2d_u8(&a.map_asf, pr.sfa, pr.k / 4, m8 / 8, pr.k / 4, 32, a.sf_groups, false));
    // 128x4 scales serve tiles that start on a 128-token boundary only.
    if (pr.sf128 && (fused || !sch.persistent || TT < 128 || pr.offsets != nullptr)) return cudaErrorInvalidValue;
    if (!ok) {
        *encode_failed = true;
        return cudaErrorInvalidValue;
    }
    const int kq = static_cast<int>(pr.k / 128);
    const int tok_tiles = static_cast<int>((pr.m + TT - 1) / TT);
    const int n_tiles = static_cast<int>(pr.n_pad / 128);
    const int splits = sch.persistent ? 1 : sch.split_k;
    const LaunchPlan lp = plan_for<TT, PIPES>(splits, sch.persistent, kq, pr.gated);
    if (lp.stages < 1) return cudaErrorInvalidConfiguration;
    // Split-K partials are staged in the pipeline stages, one slot per rank.
    if (splits > 1 &&
        static_cast<size_t>(splits) * 128 * tokens_per_owner(TT, splits) * 4 >
            static_cast<size_t>(PIPES * lp.stages) * G::kStageBytes)
        return cudaErrorInvalidConfiguration;

    a.wsf = pr.wsf;
    a.bias = static_cast<const __nv_bfloat16*>(pr.bias);
    a.y = static_cast<__nv_bfloat16*>(pr.y);
    a.offsets = pr.offsets;
    a.x = fused ? static_cast<const __nv_bfloat16*>(pr.x) : nullptr;
    a.m = static_cast<int>(pr.m);
    a.n = static_cast<int>(pr.n);
    a.n_pad = static_cast<int>(pr.n_pad);
    a.k = static_cast<int>(pr.k);
    a.kq = kq;
    a.experts = static_cast<int>(pr.experts);
    a.n_tiles = n_tiles;
    a.splits = splits;
    a.persistent = sch.persistent ? 1 : 0;
    a.asf128 = pr.sf128 ? pr.sfa : nullptr;
    a.hq = pr.gated ? pr.hq : nullptr;
    a.hsf = pr.gated ? pr.hsf : nullptr;
    a.stages = lp.stages;
    a.tmem_cols = lp.tmem_cols;
    const uint64_t wait_limit = g_wait_limit_ns.load(std::memory_order_relaxed);
    a.wait_ns = wait_limit ? wait_limit : kWaitNs;
    const size_t smem = lp.smem;

    cudaError_t err = cudaFuncSetAttribute(mxfp8_gemm_kernel<TT, PIPES, MODE>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;

    // TMEM is never oversubscribed: co-resident CTAs x columns <= 512.
    int per_sm = 1;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, mxfp8_gemm_kernel<TT, PIPES, MODE>, kThreads, smem);
    if (err != cudaSuccess) return err;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    if (static_cast<uint32_t>(per_sm) * a.tmem_cols > 512u) return cudaErrorInvalidConfiguration;
    // Persistent tiles: a second accumulator per pipe where tensor memory
    // allows it, so the next tile's MMAs overlap this tile's epilogue.
    a.acc_bufs = 1;
    if (sch.persistent) {
        const uint32_t cols2 = pow2_cols(2 * PIPES * TT + PIPES * lp.stages * G::kSfSlotCols);
        if (cols2 <= 512u && static_cast<uint32_t>(per_sm) * cols2 <= 512u) {
            a.acc_bufs = 2;
            a.tmem_cols = cols2;
        }
    }

    int grid;
    if (!sch.persistent) {
        a.num_tiles = n_tiles * tok_tiles;
        grid = a.num_tiles * splits;
    } else if (pr.offsets == nullptr) {
        a.num_tiles = n_tiles * tok_tiles;
        grid = a.num_tiles < num_sms * per_sm ? a.num_tiles : num_sms * per_sm;
    } else {
        a.num_tiles = 0;  // counted on the device from the offsets
        grid = num_sms * per_sm;
    }

    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attrs[2];
    int na = 0;
    if (splits > 1) {
        attrs[na].id = cudaLaunchAttributeClusterDimension;
        attrs[na].val.clusterDim.x = splits;
        attrs[na].val.clusterDim.y = 1;
        attrs[na].val.clusterDim.z = 1;
        ++na;
    }
    attrs[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    cfg.attrs = attrs;
    cfg.numAttrs = na;
    t_last_schedule[0] = TT + 1000 * (PIPES - 1);
    t_last_schedule[1] = sch.persistent ? -1 : splits;
    t_last_schedule[2] = fused ? 1 : 0;
    t_last_schedule[3] = grid;
    t_last_schedule[4] = lp.stages;
    return cudaLaunchKernelEx(&cfg, mxfp8_gemm_kernel<TT, PIPES, MODE>, a);
}

template <int TT, bool SF128 = false>
cudaError_t launch_dual(const GemmProblem& pr, int num_sms, cudaStream_t s, bool* encode_failed) {
    using G = DualGeometry<TT, SF128>;
    if (pr.sf128 != SF128) return cudaErrorInvalidValue;
    GemmArgs a;
    memset(&a, 0, sizeof(a));
    const int64_t m8 = (pr.m + 7) / 8 * 8;
    a.box_rows = TT;
    a.sf_groups = TT / 8 + 1;
    const bool ok = encode_2d_u8(&a.map_w, pr.wq, pr.k, pr.n_pad, pr.k, 128, 128, true) &&
                    encode_2d_u8(&a.map_a, pr.qa, pr.k, pr.m, pr.k, 128, TT, true) &&
                    (SF128 ? encode_2d(&a.map_asf, pr.sfa, CU_TENSOR_MAP_DATA_TYPE_UINT32, (pr.k / 128) * 128,
                                       (pr.m + 127) / 128, (pr.k / 128) * 512, 128, G::kRawTiles, false)
                           : encode_2d_u8(&a.map_asf, pr.sfa, pr.k / 4, m8 / 8, pr.k / 4, 32, a.sf_groups, false));
    a.asf128 = SF128 ? pr.sfa : nullptr;
    if (!ok) {
        *encode_failed = true;
        return cudaErrorInvalidValue;
    }
    a.wsf = pr.wsf;
    a.bias = static_cast<const __nv_bfloat16*>(pr.bias);
    a.y = static_cast<__nv_bfloat16*>(pr.y);
    a.m = static_cast<int>(pr.m);
    a.n = static_cast<int>(pr.n);
    a.n_pad = static_cast<int>(pr.n_pad);
    a.k = static_cast<int>(pr.k);
    a.kq = static_cast<int>(pr.k / 128);
    a.experts = 1;
    a.n_tiles = static_cast<int>(pr.n_pad / 128);
    a.splits = 1;
    a.persistent = 1;
    const int ctrl = 1024;  // barriers and the TMEM slot
    int stages = (227 * 1024 - 1024 - ctrl) / G::kStageBytes;
    if (stages > 6) stages = 6;
    if (stages < 2) return cudaErrorInvalidConfiguration;
    a.stages = stages;
    a.tmem_cols = pow2_cols(2 * TT + stages * 2 * G::kSlotCols);
    if (a.tmem_cols > 512) return cudaErrorInvalidConfiguration;
    const uint64_t wait_limit = g_wait_limit_ns.load(std::memory_order_relaxed);
    a.wait_ns = wait_limit ? wait_limit : kWaitNs;
    const size_t smem = 1024 + static_cast<size_t>(stages) * G::kStageBytes + ctrl;
    cudaError_t err = cudaFuncSetAttribute(mxfp8_gemm_dual_kernel<TT, SF128>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    int per_sm = 1;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, mxfp8_gemm_dual_kernel<TT, SF128>, kDualThreads,
                                                        smem);
    if (err != cudaSuccess) return err;
    if (per_sm < 1 || static_cast<uint32_t>(per_sm) * a.tmem_cols > 512u) return cudaErrorInvalidConfiguration;
    const int tok_tiles = static_cast<int>((pr.m + TT - 1) / TT);
    a.num_tiles = ((a.n_tiles + 1) / 2) * tok_tiles;
    const int grid = a.num_tiles < num_sms * per_sm ? a.num_tiles : num_sms * per_sm;
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kDualThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    t_last_schedule[0] = TT + 1000;
    t_last_schedule[1] = -2;  // persistent, two weight tiles per CTA tile
    t_last_schedule[2] = 0;
    t_last_schedule[3] = grid;
    t_last_schedule[4] = stages;
    return cudaLaunchKernelEx(&cfg, mxfp8_gemm_dual_kernel<TT, SF128>, a);
}

}  // namespace

std::atomic<int> g_force_pipes{0};  // testing hook, any thread; 0: automatic

void set_pipes(int pipes) {
    g_force_pipes.store((pipes == 1 || pipes == 2 || pipes == 4) ? pipes : 0, std::memory_order_relaxed);
}

GemmSchedule choose_schedule(const GemmProblem& p, int num_sms, int force_tt, int force_split,
                             int force_fuse) {
    GemmSchedule sch;
    const int64_t kq = p.k / 128;
    int tt;
    if (p.offsets != nullptr) {
        // Grouped: a token tile of at least twice the mean segment, so that
        // most experts' weights stream once (measured on the 128-expert
        // gate_up workload: 32-token tiles for a mean of 16 rows).
        const int64_t mean = (p.m + p.experts - 1) / (p.experts > 0 ? p.experts : 1);
        tt = 2 * mean <= 16 ? 16 : 2 * mean <= 32 ? 32 : 2 * mean <= 64 ? 64 : mean <= 128 ? 128 : 256;
    } else {
        // Up to 128 tokens the 64-token tile with split-K measured fastest
        // (more CTAs stream weights at once); above, persistent 256-token tiles.
        tt = p.m <= 16 ? 16 : p.m <= 32 ? 32 : p.m <= 128 ? 64 : 256;
    }
    if (force_tt) tt = force_tt;
    if (p.gated && tt > 128) tt = 128;  // the gated exchange buffer holds 64 x TT FP32
    // Dense large M: two weight tiles x TT tokens per CTA tile whenever that
    // still gives every SM a tile.  TT is the width with the least predicted
    // time, waves x the measured cost of one tile of that width (8192^3,
    // us per tile x 100; 192 runs three pipeline stages, the others four):
    // 192: 389 us in 10 waves, 176: 372 in 10, 160: 390.5 in 11, 144: 416
    // in 12.  So 176-token tiles win there (1504 tiles = 9.9 waves of 152,
    // against 1376 = 9.05 for 192).
    bool dual = false;
    int dual_tt = 192;
    if (p.offsets == nullptr && !p.gated && !p.sf128 && tt == 256 && force_tt == 0 &&
        ((p.n_pad / 128 + 1) / 2) * ((p.m + 191) / 192) >= num_sms) {
        dual = true;
        constexpr int kWidth[4] = {192, 176, 160, 144};
        constexpr int64_t kTileCost[4] = {3890, 3720, 3550, 3470};
        int64_t best = -1;
        for (int i = 0; i < 4; ++i) {
            const int w = kWidth[i];
            const int64_t tiles = ((p.n_pad / 128 + 1) / 2) * ((p.m + w - 1) / w);
            const int64_t cost = ((tiles + num_sms - 1) / num_sms) * kTileCost[i];
            if (best < 0 || cost < best) { best = cost; dual_tt = w; }
        }
    }
    if (p.offsets == nullptr && (force_tt == 192 || force_tt == 176 || force_tt == 160 || force_tt == 144)) {
        dual = true;
        dual_tt = force_tt;
    }
    if (dual) tt = dual_tt;
    bool persistent = p.offsets != nullptr || tt > 128;
    int split = 1;
    if (!persistent) {
        const int64_t tiles = (p.n_pad / 128) * ((p.m + tt - 1) / tt);
        // Measured on the decode and mid-batch shapes: as many CTAs as fit
        // two per SM (tiles of <= 64 tokens run two per SM), at least two K
        // blocks per CTA, and at most 4 per cluster -- beyond that the cluster
        // barrier and the reduction cost more than the extra streams save.
        int64_t want = ((tt <= 64 ? 2 : 1) * num_sms) / tiles;
        if (want > 4) want = 4;
        if (want > kq / 2) want = kq / 2;
        if (want < 1) want = 1;
        split = static_cast<int>(want);
    }
    if (force_split < 0 && p.offsets == nullptr && tt <= 256) {
        persistent = true;
        split = 1;
    } else if (force_split > 0 && p.offsets == nullptr && tt <= 128) {
        persistent = false;
        split = force_split;
    }
    if (split > kq) split = static_cast<int>(kq);
    bool fuse = !persistent && p.x != nullptr && p.m <= 64;
    if (force_fuse == 0) fuse = false;
    if (force_fuse == 1) fuse = !persistent && p.x != nullptr;
    sch.tokens_per_tile = tt;
    sch.split_k = persistent ? 1 : split;
    sch.persistent = persistent;
    sch.fuse_quant = fuse && !dual;
    sch.dual = dual;
    // Two MMA pipelines per CTA where the per-thread issue cost bounds the
    // stream of weights (measured): grouped tiles of <= 64 tokens; one-tile
    // schedules of <= 32 tokens (two such CTAs fit an SM); 64-token one-tile
    // schedules that still fit one CTA per SM.
    int pipes = 1;
    if (p.offsets != nullptr && tt <= 64) pipes = 2;
    // Grouped 32-token tiles: four pipelines (measured on the 128-expert
    // layer: MoE 130.7 -> 125.2 us, gate_up 71.4 -> 70.0 us against two).
    if (p.offsets != nullptr && tt == 32) pipes = 4;
    if (p.offsets == nullptr && !persistent && tt <= 32) pipes = 2;
    if (p.offsets == nullptr && !persistent && tt == 64 &&
        (p.n_pad / 128) * ((p.m + tt - 1) / tt) * split <= num_sms)
        pipes = 2;
    if (const int fp = g_force_pipes.load(std::memory_order_relaxed)) pipes = fp;
    if (pipes == 2 && tt > 64) pipes = 1;
    if (pipes == 4 && tt != 16 && tt != 32) pipes = tt <= 64 ? 2 : 1;
    if (pipes == 4 && tt == 16 && p.gated) pipes = 2;  // no four-pipe gated 16-token kernel
    sch.pipes = pipes;
    return sch;
}

cudaError_t launch_gemm(const GemmProblem& p, const GemmSchedule& sch, int num_sms, cudaStream_t s,
                        bool* encode_failed) {
    *encode_failed = false;
    if (sch.dual && p.sf128) {
        // 128x4 token scales (up to three raw scale tiles per stage, so three
        // 57 KB stages): 176-token tiles only.
        if (sch.tokens_per_tile != 176) return cudaErrorInvalidValue;
        return launch_dual<176, true>(p, num_sms, s, encode_failed);
    }
    if (sch.dual) {
        switch (sch.tokens_per_tile) {
            case 144: return launch_dual<144>(p, num_sms, s, encode_failed);
            case 160: return launch_dual<160>(p, num_sms, s, encode_failed);
            case 176: return launch_dual<176>(p, num_sms, s, encode_failed);
            default: return launch_dual<192>(p, num_sms, s, encode_failed);
        }
    }
    if (p.gated && p.sf128) return cudaErrorInvalidValue;
    if (p.gated) {  // grouped SwiGLU: tiles of <= 128 tokens
        if (sch.pipes == 2) {
            switch (sch.tokens_per_tile) {
                case 16: return launch_tt<16, 2, kModeGated>(p, sch, num_sms, s, encode_failed);
                case 32: return launch_tt<32, 2, kModeGated>(p, sch, num_sms, s, encode_failed);
                case 64: return launch_tt<64, 2, kModeGated>(p, sch, num_sms, s, encode_failed);
                default: return cudaErrorInvalidValue;
            }
        }
        if (sch.pipes == 4 && sch.tokens_per_tile == 32)
            return launch_tt<32, 4, kModeGated>(p, sch, num_sms, s, encode_failed);
        if (sch.pipes != 1) return cudaErrorInvalidValue;
        switch (sch.tokens_per_tile) {
            case 16: return launch_tt<16, 1, kModeGated>(p, sch, num_sms, s, encode_failed);
            case 32: return launch_tt<32, 1, kModeGated>(p, sch, num_sms, s, encode_failed);
            case 64: return launch_tt<64, 1, kModeGated>(p, sch, num_sms, s, encode_failed);
            case 128: return launch_tt<128, 1, kModeGated>(p, sch, num_sms, s, encode_failed);
            default: return cudaErrorInvalidValue;
        }
    }
    if (p.sf128) {  // 128x4 activation scales: one pipe, tiles of 128/256 tokens
        if (sch.pipes != 1) return cudaErrorInvalidValue;
        switch (sch.tokens_per_tile) {
            case 128: return launch_tt<128, 1, kModeSf128>(p, sch, num_sms, s, encode_failed);
            case 256: return launch_tt<256, 1, kModeSf128>(p, sch, num_sms, s, encode_failed);
            default: return cudaErrorInvalidValue;
        }
    }
    if (sch.pipes == 2) {
        switch (sch.tokens_per_tile) {
            case 16: return launch_tt<16, 2, kModePlain>(p, sch, num_sms, s, encode_failed);
            case 32: return launch_tt<32, 2, kModePlain>(p, sch, num_sms, s, encode_failed);
            case 64: return launch_tt<64, 2, kModePlain>(p, sch, num_sms, s, encode_failed);
            default: return cudaErrorInvalidValue;
        }
    }
    if (sch.pipes == 4) {
        if (sch.tokens_per_tile == 16) return launch_tt<16, 4, kModePlain>(p, sch, num_sms, s, encode_failed);
        if (sch.tokens_per_tile == 32) return launch_tt<32, 4, kModePlain>(p, sch, num_sms, s, encode_failed);
        return cudaErrorInvalidValue;
    }
    switch (sch.tokens_per_tile) {
        case 16: return launch_tt<16, 1, kModePlain>(p, sch, num_sms, s, encode_failed);
        case 32: return launch_tt<32, 1, kModePlain>(p, sch, num_sms, s, encode_failed);
        case 64: return launch_tt<64, 1, kModePlain>(p, sch, num_sms, s, encode_failed);
        case 128: return launch_tt<128, 1, kModePlain>(p, sch, num_sms, s, encode_failed);
        case 256: return launch_tt<256, 1, kModePlain>(p, sch, num_sms, s, encode_failed);
        default: return cudaErrorInvalidValue;
    }
}

void set_wait_limit_ns(uint64_t ns) { g_wait_limit_ns.store(ns, std::memory_order_relaxed); }

void last_schedule(int* out5) {
    for (int i = 0; i < 5; ++i) out5[i] = t_last_schedule[i];
}

cudaError_t read_and_clear_oob_gemm(unsigned int* out) { return read_and_clear_oob_word(out); }

cudaError_t read_and_clear_gemm_error(unsigned int* out) {
    unsigned int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(out, g_gemm_error, sizeof(unsigned int));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_gemm_error, &zero, sizeof(unsigned int));
}

}  // namespace mxk
