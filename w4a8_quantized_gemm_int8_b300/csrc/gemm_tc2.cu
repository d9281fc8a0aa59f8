// INT8 x INT8 -> INT32 GEMM with fused dequant on a pair of SMs (cta_group::2).
//
// Same function as gemm_tc.cu (Cider README, "Metal Kernel Pipeline" and
// "Quantization"): acc[m,n] = sum_k q[m,k] * wq[n,k] exactly in int32, then
//   per-channel: y = fp16(((float)acc * s_a[m]) * s_w[n])
//   per-group:   f = sum over groups g, ascending, of (float)P_g * s_w[n,g]; y = fp16(f * s_a[m])
// computed on exact fp16 images of the codes with tcgen05 kind::f16 and an
// fp32 tensor-memory accumulator folded into int32 every <= 1024 k (every
// group in per-group mode), where every partial sum is an exact integer.
//
// Pair design (B300): a cluster of two CTAs on two SMs computes one 256 x 256
// tile. Each CTA loads its own 128 token rows of A and its own 128-row half of
// the 256 weight rows of B with TMA; the even CTA's MMA thread issues
// tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16), which reads A and B from
// both CTAs' shared memory and writes each CTA's 128 x 256 fp32 accumulator
// into that CTA's tensor memory. Per SM this halves the B-operand traffic
// from L2 and the tensor core's shared-memory reads of B compared with a
// 128 x 256 single-CTA tile, and frees shared memory for a deeper ring
// (6 stages of 32 KB). Both CTAs' TMA completions land on the even CTA's
// stage barrier; the MMA commits arrive on both CTAs' barriers (multicast);
// both CTAs' epilogue warps release an accumulator buffer on the even CTA's
// barrier. Persistent: each cluster walks the tile list with a stride of the
// number of clusters. Per-channel tiles may be 256 x 192 instead (N = 192
// MMAs), when that needs no more waves over the pairs (the launcher's
// rule). Every mbarrier wait is bounded.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cstdint>
#include <cstdlib>
#include <cstring>

#include "device_common.cuh"
#include "host_once.h"
#include "kernels.h"

namespace cider {
namespace gemm2 {

constexpr int BM = 128;        // token rows per CTA (256 per pair)
constexpr int BK = 64;         // one 128-byte swizzle row of fp16
constexpr int MAX_STAGES = 8;
constexpr int A_STAGE_BYTES = BM * BK * 2;
constexpr int NUM_EPI_WARPS = 8;
constexpr int NUM_EPI_THREADS = NUM_EPI_WARPS * 32;
constexpr int NUM_ROLE_THREADS = 128;
constexpr int NUM_THREADS = NUM_ROLE_THREADS + NUM_EPI_THREADS;
constexpr int TMEM_COLS = 512;  // accumulator buffers: 2 x 256 or 4 x 128 columns
constexpr int MAX_ACC = 4;       // accumulator buffers at most
constexpr int MAX_SEG_KB = 16;  // 16 x 64 = 1024 k per exact fp32 segment
constexpr int LAUNCH_REGS = 168;
constexpr int ROLE_REGS = 40;    // TMA and MMA issue need few registers
constexpr int EPI_REGS = 232;    // running sums + loaded columns per thread
constexpr int OUT_WARP_BYTES = 32 * 32 * 2;  // output staging: 32 rows x 32 fp16 per warp
constexpr int SMEM_LIMIT = 232448;           // opt-in shared memory per block
static_assert(NUM_ROLE_THREADS * ROLE_REGS + NUM_EPI_THREADS * EPI_REGS <=
                  NUM_THREADS * LAUNCH_REGS,
              "register split exceeds the launch allocation");
constexpr uint16_t kPairMask = 0x3;
// Per-group modes: tile width and groups per accumulator buffer.
constexpr int PG_BN = 256;
constexpr int PG_GPB = 1;

// Per-instantiation tile shape. BN: output columns per pair tile (each CTA
// loads BN / 2 weight rows); GPB: groups whose partials sit side by side in
// one TMEM accumulator buffer (TMEM_COLS / (GPB * BN) buffers in flight).
// All modes run 256-wide tiles with one group per buffer (two buffers), where
// the MMA issues at its full rate. Measured on B300 (public call, per-group
// N2560 K10240, M = 4096, gs 64 / gs 128; all shapes bit-exact):
//   BN 256, GPB 1 (two buffers):   493 / 316 us  (launched)
//   BN 128, GPB 2 (two buffers):   475 / 382 us
//   BN 128, GPB 1 (four buffers):  551 / 420 us
// and at M = 1024 and 8192 the launched shape is the fastest of the three.
template <int BN, int GPB, int KPS = 1>
struct Cfg {
    static constexpr int kGroups = GPB;            // groups side by side in one buffer
    static constexpr int kBufCols = kGroups * BN;  // one TMEM accumulator buffer
    // Buffers in flight: the largest power of two that fits TMEM.
    static constexpr int kNumAcc = TMEM_COLS / kBufCols >= 4 ? 4 : TMEM_COLS / kBufCols >= 2 ? 2 : 1;
    static constexpr int kCols = BN / 2;           // columns per epilogue warp and group
    static constexpr int kChunks = kCols / 32;     // 32-column TMEM loads per warp and group
    static constexpr int kScaleSet = kGroups * kCols;  // scale floats per warp and segment
    static constexpr int kBStageBytes = (BN / 2) * BK * 2;
    // A stage holds KPS 64-k blocks of A and of B.
    static constexpr int kStageTx = 2 * KPS * (A_STAGE_BYTES + kBStageBytes);  // both CTAs
    static constexpr int kStageBytes = KPS * (A_STAGE_BYTES + kBStageBytes);
    static constexpr int kFixedBytes =
        NUM_EPI_WARPS * OUT_WARP_BYTES + NUM_EPI_WARPS * 2 * kScaleSet * 4 + 256 + 16 + 1024;
    static constexpr int kStages = (SMEM_LIMIT - kFixedBytes) / kStageBytes < MAX_STAGES
                                       ? (SMEM_LIMIT - kFixedBytes) / kStageBytes
                                       : MAX_STAGES;
    static_assert(kNumAcc * kBufCols <= TMEM_COLS && kNumAcc >= 2 && kNumAcc <= MAX_ACC &&
                      (kNumAcc & (kNumAcc - 1)) == 0 && kCols % 32 == 0,
                  "accumulator buffers fit TMEM");
    static_assert(kStages * KPS >= 6, "pipeline depth (k-blocks in flight)");
};

struct __align__(8) Barriers {
    uint64_t full[MAX_STAGES];   // even CTA: both CTAs' tile bytes landed
    uint64_t empty[MAX_STAGES];  // each CTA: the MMAs reading the stage completed
    uint64_t acc_full[MAX_ACC];   // each CTA: accumulator buffer ready
    uint64_t acc_empty[MAX_ACC];  // even CTA: both CTAs' epilogues drained the buffer
    uint64_t drain;              // even CTA: MMA drain after an abort
};
static_assert(sizeof(Barriers) <= 256, "barrier area");

template <int BN, int GPB, int KPS = 1>
struct SmemLayout {
    using C = Cfg<BN, GPB, KPS>;
    static constexpr int STAGES = C::kStages;
    static constexpr int a_off = 0;
    static constexpr int b_off = a_off + STAGES * KPS * A_STAGE_BYTES;
    static constexpr int out_off = b_off + STAGES * KPS * C::kBStageBytes;  // per-warp output staging
    // Per epilogue warp: two sets of its columns' weight scales.
    static constexpr int scale_off = out_off + NUM_EPI_WARPS * OUT_WARP_BYTES;
    static constexpr int bar_off = scale_off + NUM_EPI_WARPS * 2 * C::kScaleSet * 4;
    static constexpr int misc_off = bar_off + 256;  // tmem base, abort
    static constexpr int bytes = misc_off + 16;
    static constexpr int alloc_bytes = bytes + 1024;  // runtime 1024-byte alignment slack
    static_assert(alloc_bytes <= SMEM_LIMIT, "shared memory per block");
    static_assert(out_off % 1024 == 0, "64-byte-swizzled staging alignment");
};

struct Params {
    int M, N, K;
    int num_kb;
    int seg_kb;    // k-blocks per segment (one TMEM buffer)
    int num_seg;
    int group_kb;  // k-blocks per group (per-group; = seg_kb for per-channel)
    int G;
    int tiles_m, tiles_n;  // tiles of 256 x BN
    const float* s_a;
    const float* s_w;
    const float* s_wT;  // optional group-major copy of per-group scales [G, N]
    void* out;
    int tma_store;  // fp16 output written through tmap_y (N % 8 == 0)
    int out_bf16;   // output elements are bfloat16 instead of fp16
    uint64_t timeout_ns;
    unsigned long long* status;
};

enum : uint32_t {
    kSiteProducerEmpty = 0x301,
    kSiteMmaAccEmpty = 0x302,
    kSiteMmaFull = 0x303,
    kSiteEpiAccFull = 0x304,
    kSiteDrain = 0x305,
    kSiteProducerDrain = 0x306,
};

__device__ __forceinline__ void tile_coords(int tile, int tiles_m, int& tm, int& tn) {
    tm = tile % tiles_m;
    tn = tile / tiles_m;
}

// The four MMAs of one 64-k block on the pair (both operands advance 32 bytes
// per 16 k within their 128-byte swizzle rows), issued from one asm block;
// the first accumulates only if `accumulate`.
__device__ __forceinline__ void mma4_pair_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                              uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, t;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "setp.eq.b32 t, %4, %4;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %5, %6, %3, t;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %7, %8, %3, t;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %9, %10, %3, t;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "l"(a_desc + 2), "l"(b_desc + 2),
        "l"(a_desc + 4), "l"(b_desc + 4), "l"(a_desc + 6), "l"(b_desc + 6)
        : "memory");
}

// KPS: 64-k blocks per stage. With two (per-channel modes, and per-group
// modes whose groups are whole stages), the MMA thread
// waits and commits once per eight MMAs: tcgen05.mma holds its issuing
// thread until the tensor core takes it, so every wait, commit and loop step
// of that thread adds to a k-block's time. Params then count stages in
// num_kb and seg_kb.
template <GemmMode MODE, int BN, int GPB, int KPS>
__global__ void __cluster_dims__(2, 1, 1) __maxnreg__(LAUNCH_REGS)
    gemm_tc2_kernel(const __grid_constant__ CUtensorMap tmap_a,
                    const __grid_constant__ CUtensorMap tmap_b,
                    const __grid_constant__ CUtensorMap tmap_y, const Params p) {
    static_assert(KPS == 1 || (KPS == 2 && GPB == 1),
                  "two k-blocks per stage: one group per accumulator buffer");
    using C = Cfg<BN, GPB, KPS>;
    using SmemLayout = gemm2::SmemLayout<BN, GPB, KPS>;
    constexpr int STAGES = SmemLayout::STAGES;
    constexpr int COLS = C::kCols;
    constexpr int GS = C::kGroups;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    Barriers* bars = reinterpret_cast<Barriers*>(smem + SmemLayout::bar_off);
    float* scales = reinterpret_cast<float*>(smem + SmemLayout::scale_off);
    uint32_t* tmem_base_slot = reinterpret_cast<uint32_t*>(smem + SmemLayout::misc_off);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SmemLayout::misc_off + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();  // 0: issues the MMAs
    const int cluster = (int)cluster_id_x();
    const int nclusters = (int)num_clusters_x();
    const int num_tiles = p.tiles_m * p.tiles_n;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&bars->full[s]), 1);
            mbar_init(smem_u32(&bars->empty[s]), 1);
        }
        for (int b = 0; b < C::kNumAcc; ++b) {
            mbar_init(smem_u32(&bars->acc_full[b]), 1);
            mbar_init(smem_u32(&bars->acc_empty[b]), 2 * NUM_EPI_WARPS);
        }
        mbar_init(smem_u32(&bars->drain), 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&tmap_a);
        prefetch_tmap(&tmap_b);
        if (p.tma_store) prefetch_tmap(&tmap_y);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_base_slot), TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    // Both CTAs' barriers are initialised before any cross-CTA arrive or TMA.
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_base_slot;
    // Everything above overlaps the tail of the preceding kernel (programmatic
    // dependent launch); global memory is touched only after this wait.
    grid_dep_wait();
    grid_dep_launch();

    if (warp < 4) {
        setmaxnreg_dec<ROLE_REGS>();
        if (warp == 0 && lane == 0) {
            // ------------------------------ TMA producer (both CTAs) ----------
            int stage = 0;
            uint32_t phase = 0;
            int issued = 0;  // stage-uses issued
            for (int tile = cluster; tile < num_tiles; tile += nclusters) {
                int tm, tn;
                tile_coords(tile, p.tiles_m, tm, tn);
                const int a_row = tm * (2 * BM) + (int)rank * BM;
                const int b_row = tn * BN + (int)rank * (BN / 2);
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!mbar_wait_bounded(smem_u32(&bars->empty[stage]), phase ^ 1, p.timeout_ns,
                                           abort_flag, p.status, kSiteProducerEmpty))
                        goto producer_done;
                    const uint32_t fb_local = smem_u32(&bars->full[stage]);
                    if (rank == 0) mbar_arrive_expect_tx(fb_local, C::kStageTx);
                    const uint32_t fb = map_to_rank(fb_local, 0);
#pragma unroll
                    for (int j = 0; j < KPS; ++j) {
                        tma_load_2d_pair(smem_u32(smem + SmemLayout::a_off +
                                                  (stage * KPS + j) * A_STAGE_BYTES),
                                         &tmap_a, fb, (kb * KPS + j) * BK, a_row);
                        tma_load_2d_pair(smem_u32(smem + SmemLayout::b_off +
                                                  (stage * KPS + j) * C::kBStageBytes),
                                         &tmap_b, fb, (kb * KPS + j) * BK, b_row);
                    }
                    ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
        producer_done:
            // The MMA commits that release the last uses of each stage arrive
            // on this CTA's empty barriers; wait for them so that no arrive
            // (from the other CTA) is still in flight when this CTA exits.
            for (int u = (issued > STAGES ? issued - STAGES : 0); u < issued; ++u)
                if (!mbar_wait_drain(smem_u32(&bars->empty[u % STAGES]),
                                     (uint32_t)(u / STAGES) & 1u, p.timeout_ns))
                    report_device_error(p.status, kDevTimeout, kSiteProducerDrain);
        } else if (warp == 1 && lane == 0 && rank == 0) {
            // ------------------------------ MMA issuer (even CTA) -------------
            constexpr uint32_t idesc = idesc_f16_f32acc(2 * BM, BN);
            int stage = 0;
            uint32_t phase = 0;
            uint32_t seg_count = 0;
            bool issued_any = false;
            for (int tile = cluster; tile < num_tiles; tile += nclusters) {
                for (int seg = 0; seg < p.num_seg; ++seg, ++seg_count) {
                    const uint32_t b = seg_count % C::kNumAcc;
                    const uint32_t acc_phase = (seg_count / C::kNumAcc) & 1;
                    if (!mbar_wait_bounded(smem_u32(&bars->acc_empty[b]), acc_phase ^ 1,
                                           p.timeout_ns, abort_flag, p.status, kSiteMmaAccEmpty))
                        goto mma_done;
                    tc_fence_after();
                    const int kb0 = seg * p.seg_kb;
                    const int kb1 = min(p.num_kb, kb0 + p.seg_kb);
                    uint32_t d_tmem = tmem_base + b * C::kBufCols;
                    int gkb0 = kb0;  // first k-block of the current group
                    for (int kb = kb0; kb < kb1; ++kb) {
                        // Group j of the segment accumulates into its own BN columns.
                        if (kb - gkb0 == p.group_kb) {
                            gkb0 = kb;
                            d_tmem += BN;
                        }
                        if (!mbar_wait_bounded(smem_u32(&bars->full[stage]), phase, p.timeout_ns,
                                               abort_flag, p.status, kSiteMmaFull))
                            goto mma_done;
                        tc_fence_after();
#pragma unroll
                        for (int j = 0; j < KPS; ++j)
                            mma4_pair_f16(d_tmem,
                                          smem_desc_sw128_kmajor(smem_u32(
                                              smem + SmemLayout::a_off +
                                              (stage * KPS + j) * A_STAGE_BYTES)),
                                          smem_desc_sw128_kmajor(smem_u32(
                                              smem + SmemLayout::b_off +
                                              (stage * KPS + j) * C::kBStageBytes)),
                                          idesc, (kb > gkb0 || j > 0) ? 1u : 0u);
                        issued_any = true;
                        tc_commit_pair_multicast(smem_u32(&bars->empty[stage]), kPairMask);
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1;
                        }
                    }
                    tc_commit_pair_multicast(smem_u32(&bars->acc_full[b]), kPairMask);
                }
            }
        mma_done:
            if (*abort_flag && issued_any) {
                tc_commit_pair_multicast(smem_u32(&bars->drain), 0x1);
                if (!mbar_wait_drain(smem_u32(&bars->drain), 0, p.timeout_ns))
                    report_device_error(p.status, kDevTimeout, kSiteDrain);
            }
        }
    } else {
        setmaxnreg_inc<EPI_REGS>();
        // ------------------------------ epilogue (both CTAs) ------------------
        // Warp w (4..11) owns TMEM lanes 32 * (w % 4).. (its 32 token rows) and
        // the COLS columns [COLS * half, COLS * half + COLS) of each group's
        // accumulator, read 32 at a time.
        const int ewarp = warp - 4;
        const int quad = warp & 3;
        const int half = ewarp >> 2;
        // Output staging for the TMA store: 32 rows x 32 fp16 (64-byte rows,
        // 64-byte swizzle: chunk c of row r at chunk c ^ ((r >> 1) & 3)).
        uint8_t* stage_out = smem + SmemLayout::out_off + ewarp * OUT_WARP_BYTES;
        const uint32_t swz = (uint32_t)((lane >> 1) & 3);
        // This warp's weight scales: two sets, each [group][COLS columns] of
        // one segment. Lane l copies columns FPL * l .. FPL * l + FPL - 1 of
        // the next segment that needs them (the next segment in per-group
        // mode, the next tile's last segment in per-channel mode) one segment
        // ahead, with asynchronous copies that hold no registers; no other
        // warp reads them.
        constexpr int FPL = COLS / 32;  // scale floats per lane and group
        float* wsc = scales + ewarp * 2 * C::kScaleSet;
        uint32_t sbuf = 0;
        auto fetch_scales = [&](int tn, int seg, uint32_t buf) {
            const int n0 = tn * BN + half * COLS + FPL * lane;
#pragma unroll
            for (int j = 0; j < GS; ++j) {
                const int g = (p.G == 1) ? 0 : seg * GS + j;
                float* dst = wsc + buf * C::kScaleSet + j * COLS + FPL * lane;
                if (p.s_wT != nullptr && g < p.G && n0 + FPL - 1 < p.N && (p.N % FPL) == 0) {
                    // group-major copy: the lane's columns are contiguous bytes
                    if constexpr (FPL == 4)
                        cp_async_16(smem_u32(dst), p.s_wT + (int64_t)g * p.N + n0);
                    else
                        cp_async_8(smem_u32(dst), p.s_wT + (int64_t)g * p.N + n0);
                } else {
#pragma unroll
                    for (int i = 0; i < FPL; ++i) {
                        if (p.s_w != nullptr && g < p.G && n0 + i < p.N)
                            cp_async_4(smem_u32(dst + i), p.s_w + (int64_t)(n0 + i) * p.G + g);
                        else
                            dst[i] = 0.0f;
                    }
                }
            }
            cp_async_commit();
        };
        auto scales_ready = [&]() {
            cp_async_wait_all();
            __syncwarp();
        };
        if (cluster < num_tiles) {
            fetch_scales(cluster / p.tiles_m, (MODE == GemmMode::kPgF16) ? 0 : p.num_seg - 1, 0);
            scales_ready();
        }
        uint32_t seg_count = 0;
        bool store_pending = false;
        uint32_t acc[COLS];

        for (int tile = cluster; tile < num_tiles; tile += nclusters) {
            int tm, tn;
            tile_coords(tile, p.tiles_m, tm, tn);
            const int m_base = tm * (2 * BM) + (int)rank * BM + quad * 32;
            const int m = m_base + lane;
            const int n_half = tn * BN + half * COLS;

            if constexpr (MODE == GemmMode::kPgF16) {
#pragma unroll
                for (int j = 0; j < COLS; ++j) acc[j] = 0u;  // f = +0 before the first group
            }
            for (int seg = 0; seg < p.num_seg; ++seg, ++seg_count) {
                const uint32_t b = seg_count % C::kNumAcc;
                const uint32_t acc_phase = (seg_count / C::kNumAcc) & 1;
                const bool last_seg = (seg == p.num_seg - 1);
                const bool uses_scales = (MODE == GemmMode::kPgF16) || last_seg;
                const float* sc = wsc + sbuf * C::kScaleSet;

                // The other set was last read by this warp alone, in the
                // previous scale-consuming segment, which every lane has left.
                if (uses_scales) {
                    if (MODE == GemmMode::kPgF16 && seg + 1 < p.num_seg) {
                        fetch_scales(tn, seg + 1, sbuf ^ 1);
                    } else if (tile + nclusters < num_tiles) {
                        fetch_scales((tile + nclusters) / p.tiles_m,
                                     (MODE == GemmMode::kPgF16) ? 0 : p.num_seg - 1, sbuf ^ 1);
                    }
                }

                {
                    const bool ok = mbar_wait_bounded(smem_u32(&bars->acc_full[b]), acc_phase,
                                                      p.timeout_ns, abort_flag, p.status,
                                                      kSiteEpiAccFull);
                    if (!__all_sync(0xffffffffu, ok)) goto epi_done;
                }
                tc_fence_after();

                const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                                       b * C::kBufCols + half * COLS;
                // Batches of 32 columns over the segment's groups (ascending)
                // and the warp's column chunks; the next batch's TMEM load is
                // in flight while the current one is folded.
                {
                    constexpr int MAXB = GS * C::kChunks;
                    const int ng = (MODE == GemmMode::kPgF16 || MODE == GemmMode::kRawPgS32)
                                       ? min(GS, p.G - seg * GS)
                                       : 1;
                    const int nb = ng * C::kChunks;
                    auto col_of = [&](int bt) {
                        return (uint32_t)((bt / C::kChunks) * BN + (bt % C::kChunks) * 32);
                    };
                    uint32_t va[32], vb[32];
                    tmem_ld_32x32b_x32_ptr(t_row, va);
                    tmem_wait_ld_32(va);
#pragma unroll
                    for (int bt = 0; bt < MAXB; ++bt) {
                        if (bt >= nb) break;  // warp-uniform
                        uint32_t* v = (bt & 1) ? vb : va;
                        uint32_t* vn = (bt & 1) ? va : vb;
                        if (bt + 1 < nb) tmem_ld_32x32b_x32_ptr(t_row + col_of(bt + 1), vn);
                        const int jg = bt / C::kChunks;          // group within the segment
                        const int c0 = (bt % C::kChunks) * 32;   // column within the warp's span
                        if constexpr (MODE == GemmMode::kPcF16 || MODE == GemmMode::kRawS32) {
                            // Exact fp32 integers -> int32: the fast conversion holds
                            // below 2^22; a warp holding a larger one converts all.
                            bool big = false;
#pragma unroll
                            for (int j = 0; j < 32; ++j) big |= fabsf(__uint_as_float(v[j])) >= 4194304.0f;
                            if (__any_sync(0xffffffffu, big)) {
#pragma unroll
                                for (int j = 0; j < 32; ++j) {
                                    const int part = __float2int_rn(__uint_as_float(v[j]));
                                    acc[c0 + j] = (seg == 0) ? (uint32_t)part
                                                             : (uint32_t)((int)acc[c0 + j] + part);
                                }
                            } else {
#pragma unroll
                                for (int j = 0; j < 32; j += 2) {
                                    float t0, t1;
                                    fadd2_rn(t0, t1, __uint_as_float(v[j]), __uint_as_float(v[j + 1]),
                                             12582912.0f, 12582912.0f);
                                    const int p0 = __float_as_int(t0) - 0x4B400000;
                                    const int p1 = __float_as_int(t1) - 0x4B400000;
                                    acc[c0 + j] = (seg == 0) ? (uint32_t)p0 : (uint32_t)((int)acc[c0 + j] + p0);
                                    acc[c0 + j + 1] =
                                        (seg == 0) ? (uint32_t)p1 : (uint32_t)((int)acc[c0 + j + 1] + p1);
                                }
                            }
                        } else if constexpr (MODE == GemmMode::kPgF16) {
                            // f = f + fl(P_g * s_g), both roundings kept (ascending g;
                            // f starts at +0 for each tile, as 0 + q). Products are
                            // scalar multiplies: a packed f32x2 multiply whose only use
                            // is a packed add is contracted into a fused multiply-add.
                            const float* scc = sc + jg * COLS + c0;
#pragma unroll
                            for (int j = 0; j < 32; j += 4) {
                                const float4 s4 = *reinterpret_cast<const float4*>(scc + j);
                                const float q0 = __fmul_rn(__uint_as_float(v[j]), s4.x);
                                const float q1 = __fmul_rn(__uint_as_float(v[j + 1]), s4.y);
                                const float q2 = __fmul_rn(__uint_as_float(v[j + 2]), s4.z);
                                const float q3 = __fmul_rn(__uint_as_float(v[j + 3]), s4.w);
                                float r0, r1, r2, r3;
                                fadd2_rn(r0, r1, __uint_as_float(acc[c0 + j]), __uint_as_float(acc[c0 + j + 1]), q0, q1);
                                fadd2_rn(r2, r3, __uint_as_float(acc[c0 + j + 2]), __uint_as_float(acc[c0 + j + 3]), q2, q3);
                                acc[c0 + j] = __float_as_uint(r0);
                                acc[c0 + j + 1] = __float_as_uint(r1);
                                acc[c0 + j + 2] = __float_as_uint(r2);
                                acc[c0 + j + 3] = __float_as_uint(r3);
                            }
                        } else {  // kRawPgS32: this group's partials, straight out
                            const int n_c = n_half + c0;
                            if (m < p.M && n_c < p.N) {
                                int32_t* out = static_cast<int32_t*>(p.out) +
                                               ((int64_t)m * p.N + n_c) * p.G + seg * GS + jg;
                                const int valid = min(32, p.N - n_c);
#pragma unroll
                                for (int j = 0; j < 32; ++j)
                                    if (j < valid)
                                        out[(int64_t)j * p.G] = __float2int_rn(__uint_as_float(v[j]));
                            }
                        }
                        if (bt + 1 < nb) tmem_wait_ld_32(vn);
                    }
                }
                // This warp's reads of the buffer are complete (waited, the
                // values are in registers): release it on the even CTA's
                // barrier, one relaxed arrival per warp of both CTAs; the
                // arrival orders no memory writes.
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive_cluster_relaxed(map_to_rank(smem_u32(&bars->acc_empty[b]), 0));

                if (last_seg) {
                    if constexpr (MODE == GemmMode::kRawS32) {
                        if (m < p.M) {
                            int32_t* out = static_cast<int32_t*>(p.out) + (int64_t)m * p.N;
#pragma unroll
                            for (int j = 0; j < COLS; ++j)
                                if (n_half + j < p.N) out[n_half + j] = (int)acc[j];
                        }
                    } else if constexpr (MODE == GemmMode::kPcF16 || MODE == GemmMode::kPgF16) {
                        const float sa = (m < p.M) ? __ldg(p.s_a + m) : 0.0f;
                        bool big = false;
                        if constexpr (MODE == GemmMode::kPcF16) {
#pragma unroll
                            for (int j = 0; j < COLS; ++j) {
                                const int a = (int)acc[j];
                                big |= (a >= 4194304 || a <= -4194304);
                            }
                        }
                        const bool slow_cvt = __any_sync(0xffffffffu, big);
                        // Rounds of 32 columns: dequant, stage, TMA store.
#pragma unroll
                        for (int r = 0; r < C::kChunks; ++r) {
                            uint32_t h2[16];
#pragma unroll
                            for (int j = 0; j < 32; j += 2) {
                                const int c = r * 32 + j;
                                float y0, y1;
                                if constexpr (MODE == GemmMode::kPcF16) {
                                    const float f0 = slow_cvt ? __int2float_rn((int)acc[c])
                                                              : small_int_to_float((int)acc[c]);
                                    const float f1 = slow_cvt ? __int2float_rn((int)acc[c + 1])
                                                              : small_int_to_float((int)acc[c + 1]);
                                    const float2 s2 = *reinterpret_cast<const float2*>(sc + c);
                                    float t0, t1;
                                    fmul2_rn(t0, t1, f0, f1, sa, sa);
                                    fmul2_rn(y0, y1, t0, t1, s2.x, s2.y);
                                } else {
                                    fmul2_rn(y0, y1, __uint_as_float(acc[c]), __uint_as_float(acc[c + 1]),
                                             sa, sa);
                                }
                                h2[j / 2] = pack2_rn(y0, y1, p.out_bf16 != 0);
                            }
                            if (p.tma_store) {
                                // The staging buffer is free once the previous
                                // store from it has been read out.
                                if (store_pending && lane == 0) bulk_wait_group_read0();
                                __syncwarp();
#pragma unroll
                                for (int q = 0; q < 4; ++q)
                                    *reinterpret_cast<uint4*>(stage_out + lane * 64 +
                                                              ((q ^ swz) << 4)) =
                                        make_uint4(h2[4 * q], h2[4 * q + 1], h2[4 * q + 2],
                                                   h2[4 * q + 3]);
                                fence_proxy_async_smem();
                                __syncwarp();
                                if (lane == 0) {
                                    tma_store_2d(&tmap_y, smem_u32(stage_out), n_half + r * 32,
                                                 m_base);
                                    bulk_commit_group();
                                }
                                store_pending = true;
                            } else if (m < p.M) {
                                uint16_t* out = static_cast<uint16_t*>(p.out) + (int64_t)m * p.N;
                                const uint16_t* hh = reinterpret_cast<const uint16_t*>(h2);
#pragma unroll
                                for (int j = 0; j < 32; ++j)
                                    if (n_half + r * 32 + j < p.N) out[n_half + r * 32 + j] = hh[j];
                            }
                        }
                    }
                }

                // After the release: whatever the epilogue does between the
                // accumulator-ready wait and the release delays the MMAs two
                // segments on (two buffers). Measured at group size 64
                // (M = 4096, public call): this two-set scheme 493 us; the wait
                // moved right before the set's use 546 us; a four-set ring
                // copied three segments ahead and waited for here 515 us (549
                // with its cursor recomputed by division each segment); no
                // scale copies at all (wrong results) 461 us.
                if (uses_scales) {
                    scales_ready();
                    sbuf ^= 1;
                }
            }
        }
    epi_done:
        // Every output store has completed before the CTA exits.
        if (store_pending && lane == 0) bulk_wait_group0();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    // Neither CTA leaves (or frees tensor memory) while the other may still
    // arrive on its barriers or the MMAs may still write its tensor memory.
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

}  // namespace gemm2

namespace {

template <GemmMode MODE, int BN, int GPB, int KPS = 1>
cudaError_t launch_pair_mode(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& ty,
                             const gemm2::Params& p, int num_sms, cudaStream_t stream) {
    using namespace gemm2;
    using SmemLayout = gemm2::SmemLayout<BN, GPB, KPS>;
    auto kern = gemm_tc2_kernel<MODE, BN, GPB, KPS>;
    // Once per device: the register count the role/epilogue split assumes,
    // the shared-memory opt-in, and how many pairs fit on the GPU at once
    // (SMs pair up within a GPC).
    static PerDevice<int> max_clusters_of;
    int max_clusters = 0;
    const cudaError_t e = max_clusters_of.get([&](int& n) {
        cudaFuncAttributes fa;
        cudaError_t r = cudaFuncGetAttributes(&fa, kern);
        if (r != cudaSuccess) return r;
        if (fa.numRegs != LAUNCH_REGS) return cudaErrorInvalidConfiguration;
        r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SmemLayout::alloc_bytes);
        if (r != cudaSuccess) return r;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * (num_sms / 2), 1, 1);
        cfg.blockDim = dim3(NUM_THREADS, 1, 1);
        cfg.dynamicSmemBytes = SmemLayout::alloc_bytes;
        cfg.numAttrs = 0;  // the kernel's compile-time cluster shape (2, 1, 1) applies
        r = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
        if (r != cudaSuccess) return r;
        return n > 0 ? cudaSuccess : cudaErrorInvalidConfiguration;
    }, &max_clusters);
    if (e != cudaSuccess) return e;
    const int tiles = p.tiles_m * p.tiles_n;
    const int clusters = tiles < max_clusters ? tiles : max_clusters;
    return launch_pdl(kern, 2 * clusters, NUM_THREADS, SmemLayout::alloc_bytes, stream, ta, tb, ty, p);
}

}  // namespace

cudaError_t launch_gemm_tc_pair(const GemmArgs& a, int num_sms, cudaStream_t stream) {
    using namespace gemm2;
    if (a.M <= 0 || a.N <= 0 || a.K <= 0 || a.K % 16 != 0) return cudaErrorInvalidValue;
    if (a.M > INT32_MAX / 2 || a.N > INT32_MAX / 2 || a.K > INT32_MAX / 2)
        return cudaErrorInvalidValue;
    const bool per_group = (a.mode == GemmMode::kPgF16 || a.mode == GemmMode::kRawPgS32);
    // Tile width and groups per accumulator buffer of the mode's kernel.
    // Per-channel tiles are 256 wide, or 192 when that takes no more waves
    // over the pairs: a 192-wide tile costs about 0.9 of a 256-wide one
    // (measured; an N = 192 MMA issues close to its execution time), so it
    // pays only where the 256-wide tiles leave a ragged last wave. Measured
    // (public call): M = 1024 at N10240 K2560 (216 against 160 tiles, 3
    // waves of 74 pairs either way) 69.8 -> 67.7 us, M = 256 42.8 -> 41.1;
    // the gate|up shape M2048 N24576 (14 waves against 11) 306 -> 352 us,
    // so it stays 256 wide.
    int BN = per_group ? PG_BN : 256;
    if (a.mode == GemmMode::kPcF16) {
        const int64_t pairs = num_sms / 2 > 0 ? num_sms / 2 : 1;
        const int64_t tm = (a.M + 2 * BM - 1) / (2 * BM);
        const int64_t waves256 = (tm * ((a.N + 255) / 256) + pairs - 1) / pairs;
        const int64_t waves192 = (tm * ((a.N + 191) / 192) + pairs - 1) / pairs;
        if (waves192 <= waves256) BN = 192;
    }
    const int GS = per_group ? PG_GPB : 1;
    // Per-group layers whose groups are a multiple of 128 k take two k-blocks
    // per stage as well (one group per accumulator buffer).
    const int pg_kps = (per_group && PG_GPB == 1 && a.group_size > 0 &&
                        a.group_size % (2 * BK) == 0)
                           ? 2
                           : 1;
    CUtensorMap ta, tb, ty;
    if (encode_tmap_f16_kmajor(&ta, a.a_img, a.M, a.K, BM, BK) != CUDA_SUCCESS ||
        encode_tmap_f16_kmajor(&tb, a.b_img, a.N, a.K, BN / 2, BK) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    // fp16 output through TMA stores of 32 x 32 boxes (64-byte swizzle) when
    // the row pitch allows it (a multiple of 16 bytes); direct stores otherwise.
    const bool f16_out = (a.mode == GemmMode::kPcF16 || a.mode == GemmMode::kPgF16);
    const bool tma_store = f16_out && (a.N % 8 == 0) &&
                           (reinterpret_cast<uintptr_t>(a.out) % 16 == 0);
    memset(&ty, 0, sizeof(ty));
    if (tma_store && encode_tmap_f16_2d(&ty, a.out, a.M, a.N, 32, 32,
                                        CU_TENSOR_MAP_SWIZZLE_64B) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    Params p{};
    p.M = (int)a.M;
    p.N = (int)a.N;
    p.K = (int)a.K;
    p.num_kb = (p.K + BK - 1) / BK;
    if (per_group) {
        if (a.group_size <= 0 || a.group_size % BK != 0 || p.K % a.group_size != 0)
            return cudaErrorInvalidValue;
        if (a.group_size / BK > MAX_SEG_KB) return cudaErrorInvalidValue;  // exact fp32 partials only
        p.group_kb = a.group_size / BK;
        if (pg_kps == 2) {  // groups of a multiple of 128 k: whole stages of two k-blocks
            p.num_kb = (p.num_kb + 1) / 2;
            p.group_kb /= 2;
        }
        p.seg_kb = p.group_kb * GS;
        p.G = p.K / a.group_size;
    } else {
        // The per-channel kernels take two k-blocks per stage: k-blocks are
        // counted in stages of 128 k from here on.
        p.num_kb = (p.num_kb + 1) / 2;
        const int max_seg = MAX_SEG_KB / 2;
        const int nseg = (p.num_kb + max_seg - 1) / max_seg;
        p.seg_kb = (p.num_kb + nseg - 1) / nseg;
        p.group_kb = p.seg_kb;
        p.G = 1;
    }
    p.num_seg = (p.num_kb + p.seg_kb - 1) / p.seg_kb;
    p.tiles_m = (p.M + 2 * BM - 1) / (2 * BM);
    p.tiles_n = (p.N + BN - 1) / BN;
    p.s_a = a.s_a;
    p.s_w = a.s_w;
    p.s_wT = (per_group && a.s_wT && reinterpret_cast<uintptr_t>(a.s_wT) % 16 == 0) ? a.s_wT
                                                                                   : nullptr;
    p.out = a.out;
    p.tma_store = tma_store ? 1 : 0;
    p.out_bf16 = a.out_bf16;
    p.timeout_ns = a.timeout_ns;
    p.status = a.status;
    switch (a.mode) {
        case GemmMode::kPcF16:
            return BN == 192
                       ? launch_pair_mode<GemmMode::kPcF16, 192, 1, 2>(ta, tb, ty, p, num_sms,
                                                                       stream)
                       : launch_pair_mode<GemmMode::kPcF16, 256, 1, 2>(ta, tb, ty, p, num_sms,
                                                                       stream);
        case GemmMode::kPgF16:
            if (pg_kps == 2)
                return launch_pair_mode<GemmMode::kPgF16, PG_BN, 1, 2>(ta, tb, ty, p, num_sms,
                                                                       stream);
            return launch_pair_mode<GemmMode::kPgF16, PG_BN, PG_GPB>(ta, tb, ty, p, num_sms,
                                                                     stream);
        case GemmMode::kRawS32:
            return launch_pair_mode<GemmMode::kRawS32, 256, 1, 2>(ta, tb, ty, p, num_sms, stream);
        case GemmMode::kRawPgS32:
            if (pg_kps == 2)
                return launch_pair_mode<GemmMode::kRawPgS32, PG_BN, 1, 2>(ta, tb, ty, p, num_sms,
                                                                          stream);
            return launch_pair_mode<GemmMode::kRawPgS32, PG_BN, PG_GPB>(ta, tb, ty, p, num_sms,
                                                                        stream);
    }
    return cudaErrorInvalidValue;
}

namespace {
int engine_override() {
    static const int engine = [] {
        const char* e = getenv("CIDER_GEMM_ENGINE");
        if (e && strcmp(e, "single") == 0) return 1;
        if (e && strcmp(e, "pair") == 0) return 2;
        return 0;
    }();
    return engine;
}
}  // namespace

bool gemm_uses_pair(int64_t M) {
    const int engine = engine_override();
    return engine == 2 || (engine == 0 && M > gemm2::BM);
}

bool gemm_reads_scales_t(const GemmArgs& a, int num_sms) {
    if (a.mode != GemmMode::kPgF16) return false;
    // The same choice as launch_gemm: the raw-code pair kernel reads s_w as
    // it is; the image pair kernel and the single-SM engine read s_wT.
    if (gemm_uses_pair(a.M)) return a.b_raw == nullptr && a.b_img != nullptr;
    return !(engine_override() != 1 && gemm_tw_takes_few_tokens(a, num_sms));
}

cudaError_t launch_gemm(const GemmArgs& a, int num_sms, cudaStream_t stream) {
    if (gemm_uses_pair(a.M)) {
        // Raw weight codes: widened on chip into tensor memory; an fp16
        // weight image (cider_gemm_images): read as it is.
        if (a.b_raw) return launch_gemm_tw(a, num_sms, stream);
        if (a.b_img) return launch_gemm_tc_pair(a, num_sms, stream);
    }
    // Few tokens on raw codes: SM pairs with the weights as the MMA's M side
    // where they fill the GPU (CIDER_GEMM_ENGINE=single keeps one SM per CTA).
    if (engine_override() != 1 && gemm_tw_takes_few_tokens(a, num_sms))
        return launch_gemm_tw(a, num_sms, stream);
    return launch_gemm_tc(a, num_sms, stream);
}

}  // namespace cider
