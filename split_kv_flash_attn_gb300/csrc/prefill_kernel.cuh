// prefill_kernel.cuh -- prefill-chunk attention on the 5th-generation tensor
// cores (template; instantiated in prefill.cu and prefill_sw.cu).
//
// The only place in the path where the work is a dense contraction: nq new
// tokens x G heads of one KV head against a range of keys.  One CTA owns a
// 128-row query tile (128/G tokens x G heads of KV head k, the GQA packing) and
// one split of the key range, and walks it in 128-key tiles:
//
//   producer      : K_j, V_j tiles (128 keys x 128 d, fp16, 128-byte swizzle)
//                   into a 2-deep K ring and a 2-deep V ring.  MODE 0: one
//                   thread of a K warp and one of a V warp issue TMA tile
//                   loads over a dense fp16 region.  MODE 2: two warps copy
//                   the K rows and two the V rows of a row list by cp.async,
//                   each pair through its own ring (padding entries copy
//                   nothing and zero-fill).  MODE 1:
//                   four warps, one key row per thread, fetch q8_0 / q4_0
//                   rows through a row list or a dense range: raw segments
//                   are staged in shared memory by cp.async one tile ahead,
//                   then decoded to fp16(d*q) and stored in the same
//                   layout.
//   MMA issue     : MODE 0, one thread issues the S MMAs and a thread of
//                   another warp the PV MMAs (a thread's issue of eight MMAs
//                   takes about as long as the tensor core runs them, so one
//                   thread for both put them in series); MODE 1 and 2, one
//                   thread issues both:
//                   S_j = Q K_j^T        tcgen05.mma kind::f16, M=N=128, into
//                                        one of two TMEM S buffers (fp32).  Q
//                                        is the A operand in shared memory
//                                        (MODE 0; it runs at the same rate as
//                                        an A in tensor memory when nothing
//                                        else sits between the MMAs) or in
//                                        tensor memory (MODE 1 and 2), placed
//                                        once by the softmax warps;
//                   O  += P_j V_j        into the TMEM O accumulator; V is the
//                                        B operand in MN-major layout.
//   softmax (0-7) : two threads per query row (TMEM lane), 64 key columns
//                   each: tcgen05.ld S_j, causal / padding mask, online
//                   softmax in log2 units, P_j (fp16) into tensor memory,
//                   where the PV MMA reads it as its A operand.  O is
//                   rescaled in TMEM only when a row maximum grows by more than
//                   2^8 (the stale maximum stays the reference otherwise,
//                   exactly as in the plain online softmax with another shift),
//                   so the softmax waits for the previous PV only then.
//                   MODE 1 and 2: an S buffer is released as soon as the
//                   softmax warps have loaded it (S_{j+1} and S_{j+2} are
//                   computed while P_j is), the row maximum is exchanged
//                   between a row's two warps before the exponentials, and
//                   P_j is written once PV_{j-1} is done.  MODE 0: two P
//                   buffers (the tensor-memory columns Q would take), so P_j
//                   is written once PV_{j-2} has read P_{j-2} and published
//                   after the next tile's scores are loaded; the exponentials
//                   are taken against the current reference while the
//                   maximum exchange completes, and taken again (the scores
//                   reloaded, the S buffer released only then) by a warp whose
//                   row's reference moves.
//
// The per-split result (O normalised, lse) is merged across splits by the
// last CTA of each (sequence, KV head, query tile), as in the decode kernel.
// Grid: x = (KV head, query tile), y = sequence, z = split, so that every CTA
// of a split is dispatched before any CTA of the next (a long head split on
// the SMs the query tiles fill, short tail splits on the SMs they leave).
// Every mbarrier wait is bounded; a wait that gives up sets the handle's
// device status word and the CTA stops issuing work, drains what it issued
// and frees its TMEM.
#pragma once

#include <string.h>

#include "internal.h"
#include "ptx.cuh"
#include "tc.cuh"

namespace skv {
namespace pf {

constexpr int kPM = 128;        // query rows per tile (TMEM lanes)
constexpr int kPN = 128;        // keys per tile
constexpr int kPD = 128;        // head dim
constexpr int kSoftmaxWarps = 8;   // two warps per query-row group (one per column half)
constexpr int kSoftmaxThreads = kSoftmaxWarps * 32;
constexpr int kTileBytes = kPN * kPD * 2;       // 32 KiB per K or V tile
constexpr int kHalfTile = kTileBytes / 2;       // one 64-column swizzle block
constexpr int kOffK = 0;                        // 2 stages (quantised keys: hi and lo of one stage)
constexpr int kOffV = kOffK + 2 * kTileBytes;   // 2 stages
// TMA instance (MODE 0): Q (the S MMA's A operand) after the V stages, then
// the barriers.  Software-producer instances keep Q in tensor memory and put
// the barriers right after the V stages; the quantised ones then stage raw
// row segments (two tiles of K and V segments), so that a tile's global
// loads are in flight while the previous tile is decoded.
constexpr int kOffQ = kOffV + 2 * kTileBytes;
constexpr int kOffBar = kOffQ;                  // software-producer instances
constexpr int kOffBarQ = kOffQ + kTileBytes;    // TMA instance
constexpr int kSmem = kOffBar + 256 + 1024;     // + barriers + alignment slack
constexpr int kOffRaw = kOffBar + 256;
__host__ __device__ constexpr int seg_bytes_of(int t) { return t == SKV_F16 ? 256 : (t == SKV_Q8_0 ? 136 : 72); }
template <int MODE, int KT, int VT>
__host__ __device__ constexpr int smem_bytes()
{
    return MODE == 0 ? kOffBarQ + 256 + 1024
                     : kSmem + (KT == SKV_F16 ? 0 : 2 * kPN * (seg_bytes_of(KT) + seg_bytes_of(VT)));
}
static_assert(kSmem + 2 * kPN * (136 + 136) <= 227 * 1024, "shared memory per CTA");
static_assert(kOffBarQ + 256 + 1024 <= 227 * 1024, "shared memory per CTA");
constexpr uint32_t kIdescS = tc::idesc_f16(kPM, kPN, false);
constexpr uint32_t kIdescPV = tc::idesc_f16(kPM, kPD, true);
constexpr float kRescaleLog2 = 8.0f;            // rescale O only when the max grows by > 2^8

// fp16 row lists (MODE 2): warps per operand, and how many of a lane's copy
// instructions for tile j go out before tile j-1 is published (the rest
// follow).  Measured on 8 x 64 tokens over 32768 listed rows: one warp per
// operand 0.59 ms, two 0.50 ms with all 32 copies first; then 16 first 0.41
// ms, 8 first 0.41 ms, none first (one tile in flight) 0.46 ms.  Three warps
// per operand (rows 44/44/40) measured 0.41 ms too; four would cap every
// thread at 96 registers.
constexpr int kRowWarps = 2;
constexpr int kPubAfter = 16;
// Producer warps and thread count per mode (MODE 0: TMA tiles, MODE 1:
// quantised rows converted by software, MODE 2: fp16 row lists by cp.async).
template <int MODE>
struct Cfg {
    // MODE 0: 12 warps, 3 per SM sub-partition, so the softmax warps keep
    // up to 168 registers; one warp streams K tiles and one V tiles, so
    // neither waits behind the other's ring slot (two lanes of one warp would
    // share its issue).  MODE 1 and 2: 13 warps, four of them producers (MODE
    // 1: each thread fetches and converts one key row of a tile; MODE 2: two
    // warps copy K rows and two V rows); the sub-partition holding four warps
    // caps every thread at 128 registers, and the producers' throughput is
    // worth more than the softmax's spare registers (two producer warps: 1.6x
    // the kernel time).
    static constexpr int kProducerWarps = MODE == 0 ? 2 : (MODE == 1 ? 4 : 2 * kRowWarps);
    // MMA issue: MODE 0, one warp for S = Q K^T and one for O += P V; the
    // software-producer modes, one warp for both (a fourteenth warp measured
    // 2 % slower there).
    static constexpr bool kSplitIssue = MODE == 0;
    static constexpr int kMmaWarp = kSoftmaxWarps + kProducerWarps;
    static constexpr int kPvWarp = kMmaWarp + (kSplitIssue ? 1 : 0);
    static constexpr int kThreads = (kPvWarp + 1) * 32;
    // arrivals that fill a K or V stage: the TMA thread's expect-tx, every
    // producer thread (MODE 1), or the threads of the operand's two warps
    static constexpr uint32_t kFullCount = MODE == 0 ? 1 : (MODE == 1 ? kProducerWarps * 32 : kRowWarps * 32);
    // arrivals on a row-list padding mask: the producer threads, or (MODE 2)
    // the two K warps
    static constexpr uint32_t kMaskCount = MODE == 2 ? kRowWarps * 32 : kProducerWarps * 32;
};

// barrier slots (8 bytes each) inside the barrier area
// Tensor memory: kSBuf S buffers (fp32), then two 64-column slots and O
// (fp32).  TMA instance: the slots are two P buffers (fp16 pairs), tile j's
// P in slot j % 2, so a tile's P is written while PV of the previous tile
// still reads its own; Q is in shared memory.  Software-producer instances
// (quantised raw staging leaves no shared memory for Q, and over row lists
// the shared-memory Q measured 2 % slower): slot 0 holds P, slot 1 Q (row m
// in lane m, dims 2c, 2c+1 in column c).  S full (MMA commit) and S free
// (the softmax warps have loaded S) are per S buffer: tile j's are buffer
// j % kSBuf, phase j / kSBuf.  P full (softmax) and P free (commit after PV:
// P read, O updated) are per P buffer: tile j's are buffer j % 2, phase j / 2
// (software producers: buffer 0, phase j).  No waiter can be two phases away from the
// phase it waits for (mbarrier waits are by phase parity), because each side
// needs the other's next step before it can complete another phase.  A commit
// arrives once every earlier MMA of the issuing thread is done, so "PV of
// tile j done" means every earlier PV is.
constexpr int kSBuf = 2;
constexpr int kPCol = kSBuf * kPN;              // P: keys 2c, 2c+1 of the tile in column kPCol (+64) + c
constexpr int kQCol = kPCol + kPN / 2;          // software-producer instances
constexpr int kOCol = kQCol + kPD / 2;          // first TMEM column of O
// (M full: row-list mode, a tile's padding mask is in shared memory; 4 slots,
// tile j in slot j % 4.)
enum { B_KFULL = 0, B_KEMPTY = 2, B_VFULL = 4, B_VEMPTY = 6, B_QFULL = 8, B_SFULL = 9, B_SFREE = 9 + kSBuf,
       B_PFULL = 9 + 2 * kSBuf, B_PFREE = 11 + 2 * kSBuf, B_MFULL = 13 + 2 * kSBuf, B_COUNT = 17 + 2 * kSBuf };
static_assert(B_COUNT * 8 <= 256, "barrier area");
static_assert(kOCol + kPD <= 512, "tensor memory columns");

struct PrefillArgs {
    const __half *q;          // [S][nq][H][D]
    int S, nq, H, Hk, G;
    float scale_log2;
    const int32_t *q_pos;     // [S][nq] or null
    int64_t key_pos0;
    int64_t logical0;
    int64_t row0;             // row of local key 0 (dense ranges)
    int64_t n_local;
    int m_tiles;
    int n_splits;
    int64_t split_len;
    float *o_split;
    float *lse_split;
    int *counters;
    float *o_out;
    float *lse_out;
    int64_t R;
    int *status;
    // software producers
    const uint8_t *k;         // region bases
    const uint8_t *v;
    int64_t k_row_bytes;
    int64_t v_row_bytes;
    const int32_t *rows;      // row lists or null (dense)
    int64_t rows_ld;
    int64_t rows_off;         // list entry of local key 0
    int rows_per_head;
};

// Byte offset of 16-byte chunk c (values 8c .. 8c+7) of key row r in a
// 128-key x 128-value fp16 tile with the 128-byte swizzle (the layout a TMA
// load of two 64-value boxes writes).
__device__ __forceinline__ uint32_t tile_off(int r, int c)
{
    return static_cast<uint32_t>((c >> 3) * kHalfTile + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// Two code bytes of a word (byte pair at bit 16*hi) -> half2(1024 + b0, 1024 + b1).
template <int HI>
__device__ __forceinline__ __half2 code_pair(uint32_t w)
{
    const uint32_t h = __byte_perm(w, 0x64646464u, HI ? 0x4342 : 0x4140);
    return *reinterpret_cast<const __half2 *>(&h);
}

// Raw bytes of a q8_0 / q4_0 head segment as 32-bit words.
template <int T>
struct QSeg {
    static constexpr int SEG = T == SKV_Q8_0 ? 136 : 72;   // 4 blocks of 34 or 18 bytes
    static constexpr int NW = SEG / 4;
};

// Write one key row of a tile from its loaded segment words: every value d*q
// as fp16, 16 swizzled 16-byte chunks per row (zeros for a padding row).
// With LO (keys), the value is split exactly into hi = fp16(d*q) in `tile`
// and lo = fp16(d*q - hi) in `tile_lo` (one fused multiply-add: d*q has at
// most 18 significant bits, so hi + lo is d*q whenever lo is a normal fp16);
// without LO (values) only fp16(d*q) is written, rounded once.
template <int T, bool LO = false>
__device__ __forceinline__ void store_row(const uint32_t (&w)[QSeg<T>::NW], bool valid, uint8_t *tile, int r,
                                          uint8_t *tile_lo = nullptr)
{
    constexpr int SEG = QSeg<T>::SEG;
    if (!valid) {
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            *reinterpret_cast<uint4 *>(tile + tile_off(r, c)) = make_uint4(0, 0, 0, 0);
            if (LO) *reinterpret_cast<uint4 *>(tile_lo + tile_off(r, c)) = make_uint4(0, 0, 0, 0);
        }
        return;
    }
    // a byte pair at even offset o lives in word o/4, half (o/2)&1
#define SKV_PAIR_WORD(o) w[(o) >> 2]
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        constexpr int BLK = SEG / 4;
        const int o_d = b * BLK;
        const uint32_t dw = SKV_PAIR_WORD(o_d);
        const __half d = __ushort_as_half(static_cast<unsigned short>((o_d & 2) ? (dw >> 16) : (dw & 0xffff)));
        const __half2 dd = __half2half2(d);
        if constexpr (T == SKV_Q8_0) {
            const __half2 bias = __half2half2(__ushort_as_half(0x6480));   // 1152 = 1024 + 128
#pragma unroll
            for (int c = 0; c < 4; ++c) {            // values 8c .. 8c+7 of the block
                uint32_t out[4], out_lo[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int o = o_d + 2 + 8 * c + 2 * i;
                    const uint32_t x = SKV_PAIR_WORD(o) ^ 0x80808080u;   // int8 q -> byte q + 128
                    const __half2 qv = __hsub2((o & 2) ? code_pair<1>(x) : code_pair<0>(x), bias);
                    const __half2 val = __hmul2(qv, dd);
                    out[i] = *reinterpret_cast<const uint32_t *>(&val);
                    if (LO) {
                        const __half2 lo = __hfma2(qv, dd, __hneg2(val));
                        out_lo[i] = *reinterpret_cast<const uint32_t *>(&lo);
                    }
                }
                *reinterpret_cast<uint4 *>(tile + tile_off(r, 4 * b + c)) = make_uint4(out[0], out[1], out[2], out[3]);
                if (LO)
                    *reinterpret_cast<uint4 *>(tile_lo + tile_off(r, 4 * b + c)) =
                        make_uint4(out_lo[0], out_lo[1], out_lo[2], out_lo[3]);
            }
        } else {
            const __half2 bias = __half2half2(__ushort_as_half(0x6408));   // 1032 = 1024 + 8
#pragma unroll
            for (int c = 0; c < 4; ++c) {            // c 0,1: low nibbles of bytes 0-7, 8-15; c 2,3: high
                uint32_t out[4], out_lo[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int o = o_d + 2 + 8 * (c & 1) + 2 * i;
                    const uint32_t raw = SKV_PAIR_WORD(o);
                    const uint32_t x = (c & 2) ? ((raw >> 4) & 0x0F0F0F0Fu) : (raw & 0x0F0F0F0Fu);
                    const __half2 qv = __hsub2((o & 2) ? code_pair<1>(x) : code_pair<0>(x), bias);
                    const __half2 val = __hmul2(qv, dd);
                    out[i] = *reinterpret_cast<const uint32_t *>(&val);
                    if (LO) {
                        const __half2 lo = __hfma2(qv, dd, __hneg2(val));
                        out_lo[i] = *reinterpret_cast<const uint32_t *>(&lo);
                    }
                }
                *reinterpret_cast<uint4 *>(tile + tile_off(r, 4 * b + c)) = make_uint4(out[0], out[1], out[2], out[3]);
                if (LO)
                    *reinterpret_cast<uint4 *>(tile_lo + tile_off(r, 4 * b + c)) =
                        make_uint4(out_lo[0], out_lo[1], out_lo[2], out_lo[3]);
            }
        }
    }
#undef SKV_PAIR_WORD
}


template <int MODE, int KT, int VT>
__global__ void __launch_bounds__(Cfg<MODE>::kThreads, 1)
    splitkv_prefill_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                           const PrefillArgs a)
{
    using C = Cfg<MODE>;
    // Quantised keys: one K stage holding the (hi, lo) pair of fp16 tiles in
    // the two K slots, and S = Q hi^T + Q lo^T (16 k-steps), so that scores
    // use the exact key values; fp16 keys: a 2-deep K ring.
    constexpr bool KLO = KT != SKV_F16;
    constexpr bool P2 = MODE == 0;              // two P buffers, Q in shared memory
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_addr(sm);
    const uint32_t bar0 = sbase + (P2 ? kOffBarQ : kOffBar);
    auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;
    __shared__ int s_maxpos;
    __shared__ int s_last;
    // [slot][column half][row]: partial row maxima by tile parity (slots 0, 1),
    // then the halves' row sums (slot 2, so that no partner read is pending)
    __shared__ float s_pair[3][2][kPM];
    // row-list mode: key-present bits of a tile (word w: keys 32w .. 32w+31), 4 slots
    __shared__ uint32_t s_vmask[4][kPN / 32];

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int mt = blockIdx.x % a.m_tiles;
    const int kh = blockIdx.x / a.m_tiles;
    const int split = blockIdx.z;
    const int s = blockIdx.y;
    const int unit = (s * a.Hk + kh) * a.m_tiles + mt;
    const int tpt = kPM / a.G;                       // tokens per query tile
    const int64_t list = a.rows_per_head ? static_cast<int64_t>(s) * a.Hk + kh : s;
    const int32_t *lrow = a.rows ? a.rows + list * a.rows_ld + a.rows_off : nullptr;   // entry of local key 0

    const int64_t j_lo = static_cast<int64_t>(split) * a.split_len;
    const int64_t j_hi = min(a.n_local, j_lo + a.split_len);

    // Softmax threads: query row m = TMEM lane (warp % 4) * 32 + lane, and the
    // column half hf (key columns hf*64 .. hf*64+63 of each 128-key tile).
    const bool softmax = warp < kSoftmaxWarps;
    const int m = (warp & 3) * 32 + lane;
    const int hf = warp >> 2;
    const int t_row = mt * tpt + m / a.G;
    const bool row_ok = softmax && t_row < a.nq;
    const int32_t pos_row = (row_ok && a.q_pos) ? a.q_pos[static_cast<int64_t>(s) * a.nq + t_row] : INT32_MAX;

    if (tid == 0) {
        s_abort = 0;
        s_maxpos = INT32_MIN;
    }
    __syncthreads();
    if (a.q_pos && row_ok && hf == 0) atomicMax(&s_maxpos, pos_row);
    if (warp == 0) {
        tc::tmem_alloc<512>(smem_addr(&s_tmem));
        tc::tmem_relinquish();
    }
    if (tid == kSoftmaxThreads) {
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(bar(B_KFULL + i), C::kFullCount);
            tc::mbar_init(bar(B_KEMPTY + i), 1);
            tc::mbar_init(bar(B_VFULL + i), C::kFullCount);
            tc::mbar_init(bar(B_VEMPTY + i), 1);
        }
        for (int i = 0; i < kSBuf; ++i) {
            tc::mbar_init(bar(B_SFULL + i), 1);
            tc::mbar_init(bar(B_SFREE + i), kSoftmaxThreads);   // S buffer free: the softmax warps loaded it
        }
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(bar(B_PFULL + i), kSoftmaxThreads);
            tc::mbar_init(bar(B_PFREE + i), 1);                  // PV of the buffer's last P done
        }
        tc::mbar_init(bar(B_QFULL), kSoftmaxThreads);
        for (int i = 0; i < 4; ++i) tc::mbar_init(bar(B_MFULL + i), C::kMaskCount);
        tc::fence_barrier_init();
        if (MODE == 0) {
            tc::prefetch_tmap(&tmap_k);
            tc::prefetch_tmap(&tmap_v);
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = s_tmem;

    // Keys past the largest query position of the tile are invisible to all
    // its rows: the tile walk stops there.
    int64_t j_end = j_hi;
    if (a.q_pos) {
        const int64_t last_visible = static_cast<int64_t>(s_maxpos) - a.key_pos0 - a.logical0;   // local index
        j_end = min(j_end, last_visible + 1);
    }
    const int n_tiles = j_end > j_lo ? static_cast<int>((j_end - j_lo + kPN - 1) / kPN) : 0;

    auto fail_wait = [&]() {
        s_abort = 1;
        if (a.status) atomicOr(a.status, 1);
    };
    // A phase already complete is taken at once: the abort flag is read only
    // when the barrier is not ready (reading it first on every wait put a
    // shared-memory round trip on each hand-off of the tile chain: 237 ->
    // 220 us on the prefill chunk's window, 645 -> 615 us over q8_0 / q4_0
    // rows).  The row-list instance keeps the flag first (341 against 367 us
    // the other way round).
    auto wait = [&](int b, uint32_t parity) -> bool {
        if (MODE != 2 && tc::mbar_try_wait(bar(b), parity)) return true;
        if (*reinterpret_cast<volatile int *>(&s_abort)) return false;
        if (tc::mbar_wait(bar(b), parity, a.status)) return true;
        fail_wait();
        return false;
    };
    // The two warps that share rows (w and w + 4) meet on named barrier 1 + w%4.
    auto pair_sync = [&]() { asm volatile("bar.sync %0, 64;\n" ::"r"(1 + (warp & 3)) : "memory"); };

    float m_ref = -INFINITY, l_run = 0.f;

    if (warp >= kSoftmaxWarps && warp < C::kMmaWarp) {
        if constexpr (MODE == 0) {
            // ---------------- TMA producer --------------------------------
            // The first producer warp streams K tiles and the second V tiles,
            // each waiting only for its own ring slot: a K load never waits
            // for a PV to finish.
            if (lane == 0) {
                const bool is_v = warp == kSoftmaxWarps + 1;
                const int b_empty = is_v ? B_VEMPTY : B_KEMPTY, b_full = is_v ? B_VFULL : B_KFULL;
                const uint32_t off = is_v ? kOffV : kOffK;
                const CUtensorMap *map = is_v ? &tmap_v : &tmap_k;
                int issued = 0;
                for (int j = 0; j < n_tiles; ++j) {
                    const int b = j & 1;
                    const int y = static_cast<int>(a.row0 + j_lo + static_cast<int64_t>(j) * kPN);
                    const int x = kh * kPD;
                    if (j >= 2 && !wait(b_empty + b, ((j >> 1) - 1) & 1)) break;
                    tc::mbar_expect_tx(bar(b_full + b), kTileBytes);
                    tc::tma_load_2d(sbase + off + b * kTileBytes, map, x, y, bar(b_full + b));
                    tc::tma_load_2d(sbase + off + b * kTileBytes + kHalfTile, map, x + 64, y, bar(b_full + b));
                    ++issued;
                }
                if (*reinterpret_cast<volatile int *>(&s_abort)) {
                    // drain: every issued load must land before the CTA exits
                    for (int j = (issued > 2 ? issued - 2 : 0); j < issued; ++j)
                        tc::mbar_wait(bar(b_full + (j & 1)), (j >> 1) & 1, nullptr, 100000000ull);
                }
            }
        } else if constexpr (MODE == 2) {
            // ---------------- fp16 row lists: two K warps, two V warps -------
            // Each pair streams its own operand through its 2-slot ring, as
            // the TMA warps do: tile j's copies are issued once its slot is
            // free, and tile j-1 is published when its copies have landed, so
            // up to two tiles of each operand are in flight and a K tile never
            // waits for a PV.  A warp copies 64 rows of a tile, two rows per
            // cp.async instruction (16 lanes x 16 bytes cover one row's 256
            // bytes, so an instruction touches four cache lines); lane l holds
            // the list entries of its rows l and l + 32.  Padding entries copy
            // nothing (source size 0 zero-fills).  The K warps publish each
            // tile's padding mask when they issue it: its slot (j % 4) was last
            // read by the softmax of tile j - 4, before P(j - 4) was published,
            // and PV(j - 4) is issued before S(j - 2), whose completion freed
            // the K slot.
            static_assert(KT == SKV_F16 && VT == SKV_F16, "fp16 rows");
            constexpr int W = kRowWarps;               // warps per operand
            constexpr int RW = kPN / W;                   // rows a warp copies
            constexpr int NH = RW / 32;                   // list entries a lane holds
            const int pw = warp - kSoftmaxWarps;          // 0 .. W-1: K; W .. 2W-1: V
            const bool is_v = pw >= W;
            const int rbase = (pw % W) * RW;              // first tile row of this warp
            const uint8_t *base = is_v ? a.v : a.k;
            const int64_t row_bytes = is_v ? a.v_row_bytes : a.k_row_bytes;
            const uint8_t *seg0 = base + static_cast<int64_t>(kh) * (kPD * 2) + 16 * (lane & 15);
            const uint32_t ring = sbase + (is_v ? kOffV : kOffK);
            const int b_empty = is_v ? B_VEMPTY : B_KEMPTY, b_full = is_v ? B_VFULL : B_KFULL;
            auto entry = [&](int j, int h) -> int {
                const int64_t key = j_lo + static_cast<int64_t>(j) * kPN + rbase + 32 * h + lane;
                return (j < n_tiles && key < j_hi) ? __ldg(lrow + key) : -1;
            };
            int cur[NH], nxt[NH];
#pragma unroll
            for (int h = 0; h < NH; ++h) cur[h] = entry(0, h);
            int issued = 0;
            for (int j = 0; j < n_tiles; ++j) {
                const int b = j & 1;
#pragma unroll
                for (int h = 0; h < NH; ++h) nxt[h] = entry(j + 1, h);
                if (!__all_sync(0xffffffffu, j < 2 || wait(b_empty + b, ((j >> 1) - 1) & 1))) break;
                if (!is_v) {
                    const int64_t key = j_lo + static_cast<int64_t>(j) * kPN + rbase + lane;
#pragma unroll
                    for (int h = 0; h < NH; ++h) {
                        const uint32_t w = __ballot_sync(0xffffffffu, cur[h] >= 0 || key + 32 * h >= j_hi);
                        if (lane == 0) s_vmask[j & 3][rbase / 32 + h] = w;
                    }
                    __syncwarp();
                    tc::mbar_arrive(bar(B_MFULL + (j & 3)));
                }
                const uint32_t tile_s = ring + static_cast<uint32_t>(b * kTileBytes);
                auto copy = [&](int it) {
                    const int rr = 2 * it + (lane >> 4);      // row of this warp's RW
                    const int row = __shfl_sync(0xffffffffu, cur[it / 16], rr & 31);
                    cp_async16(tile_s + tile_off(rbase + rr, lane & 15),
                               row >= 0 ? seg0 + static_cast<int64_t>(row) * row_bytes : base, row >= 0 ? 16 : 0);
                };
                // The first PUB copy instructions of tile j go out before tile
                // j-1 is published (so that the S MMA of tile j-1 does not wait
                // for all of them), the rest after.
                constexpr int PUB = kPubAfter;
                if (PUB > 0) {
#pragma unroll
                    for (int it = 0; it < PUB; ++it) copy(it);
                    cp_async_commit();
                }
                if (j >= 1) {
                    if (PUB > 0) cp_async_wait<1>();          // this thread's copies of tile j-1
                    else cp_async_wait<0>();
                    tc::fence_proxy_async_smem();
                    tc::mbar_arrive(bar(b_full + ((j - 1) & 1)));
                }
#pragma unroll
                for (int it = PUB; it < RW / 2; ++it) copy(it);
                cp_async_commit();
                ++issued;
#pragma unroll
                for (int h = 0; h < NH; ++h) cur[h] = nxt[h];
            }
            cp_async_wait<0>();
            if (issued == n_tiles && issued > 0) {
                tc::fence_proxy_async_smem();
                tc::mbar_arrive(bar(b_full + ((issued - 1) & 1)));
            }
        } else {
            // ---------------- quantised rows: kPN / NPT key rows a thread -----
            // No wait may depend on a tile the producers have not published yet.
            static_assert(KT != SKV_F16 && VT != SKV_F16, "quantised rows");
            constexpr int NPT = C::kProducerWarps * 32;      // producer threads
            constexpr int RPT = kPN / NPT;                   // rows per thread
            const int r0 = tid - kSoftmaxThreads;
            constexpr int SEGK = seg_bytes_of(KT), SEGV = seg_bytes_of(VT);
            // Cache row of key row r0 + u*NPT of tile j (-1: padding or past
            // the split).
            auto tile_row = [&](int j, int u) -> int64_t {
                const int64_t key = j_lo + static_cast<int64_t>(j) * kPN + r0 + u * NPT;
                if (key >= j_hi) return -1;
                return lrow ? static_cast<int64_t>(__ldg(lrow + key)) : a.row0 + key;
            };
            auto k_src = [&](int64_t row) {
                return row >= 0 ? a.k + row * a.k_row_bytes + static_cast<int64_t>(kh) * SEGK : nullptr;
            };
            auto v_src = [&](int64_t row) {
                return row >= 0 ? a.v + row * a.v_row_bytes + static_cast<int64_t>(kh) * SEGV : nullptr;
            };
            // Row-list mode: tile j's key-present bits (a list row, or past the
            // split, masked there) to shared memory for the softmax.
            auto publish_mask = [&](int j, const int64_t (&rw)[RPT]) {
                if (!lrow) return;
                uint32_t present[RPT];
#pragma unroll
                for (int u = 0; u < RPT; ++u) {
                    const int64_t key = j_lo + static_cast<int64_t>(j) * kPN + r0 + u * NPT;
                    present[u] = __ballot_sync(0xffffffffu, rw[u] >= 0 || key >= j_hi);
                }
                if ((tid & 31) == 0) {
#pragma unroll
                    for (int u = 0; u < RPT; ++u) s_vmask[j & 3][(r0 + u * NPT) >> 5] = present[u];
                }
                __syncwarp();
                tc::mbar_arrive(bar(B_MFULL + (j & 3)));
            };
            // Each thread's raw segments of tile j+1 are copied
            // (cp.async, 8-byte pieces) into a staging slot while tile j is
            // decoded from the other slot into the fp16 operand tiles.  A
            // thread decodes exactly the rows it staged, so its own copy
            // groups order everything; list entries run two tiles ahead.
            uint8_t *raw = sm + kOffRaw;
            constexpr int RAWK = kPN * SEGK, RAWV = kPN * SEGV;
            auto raw_k = [&](int slot, int r) { return raw + slot * (RAWK + RAWV) + r * SEGK; };
            auto raw_v = [&](int slot, int r) { return raw + slot * (RAWK + RAWV) + RAWK + r * SEGV; };
            auto issue_raw = [&](int slot, const int64_t (&rw)[RPT]) {
#pragma unroll
                for (int u = 0; u < RPT; ++u) {
                    const int r = r0 + u * NPT;
                    const uint8_t *ks = k_src(rw[u]);
                    const uint8_t *vs = v_src(rw[u]);
#pragma unroll
                    for (int i = 0; i < SEGK / 8; ++i)
                        cp_async8(smem_addr(raw_k(slot, r) + 8 * i), ks ? ks + 8 * i : a.k, ks ? 8 : 0);
#pragma unroll
                    for (int i = 0; i < SEGV / 8; ++i)
                        cp_async8(smem_addr(raw_v(slot, r) + 8 * i), vs ? vs + 8 * i : a.v, vs ? 8 : 0);
                }
                cp_async_commit();
            };
            int64_t e0[RPT], e1[RPT];
#pragma unroll
            for (int u = 0; u < RPT; ++u) {
                e0[u] = n_tiles > 0 ? tile_row(0, u) : -1;
                e1[u] = n_tiles > 1 ? tile_row(1, u) : -1;
            }
            if (n_tiles > 0) issue_raw(0, e0);
            for (int j = 0; j < n_tiles; ++j) {
                const int b = j & 1;
                const int kb = KLO ? 0 : b;                      // K stage of this tile
                const int slot = j & 1;
                if (j + 1 < n_tiles) issue_raw(slot ^ 1, e1);
                int64_t e2[RPT];
#pragma unroll
                for (int u = 0; u < RPT; ++u) e2[u] = j + 2 < n_tiles ? tile_row(j + 2, u) : -1;
                if (j + 1 < n_tiles) cp_async_wait<1>();        // this thread's segments of tile j landed
                else cp_async_wait<0>();
                const bool k_ok = KLO ? (j < 1 || wait(B_KEMPTY, (j - 1) & 1))
                                      : (j < 2 || wait(B_KEMPTY + b, ((j >> 1) - 1) & 1));
                if (!__all_sync(0xffffffffu, k_ok)) break;
                // The mask slot of tile j is free here: S(j-1) is issued
                // after PV(j-3), and so after the softmax of tile j-3 (and
                // of j-4) has read its mask.  K is published as soon as it
                // is stored, so S(j) never waits for the V slot.
                publish_mask(j, e0);
#pragma unroll
                for (int u = 0; u < RPT; ++u) {
                    const int r = r0 + u * NPT;
                    uint32_t w[QSeg<KT>::NW];
#pragma unroll
                    for (int i = 0; i < QSeg<KT>::NW; ++i) w[i] = *reinterpret_cast<const uint32_t *>(raw_k(slot, r) + 4 * i);
                    store_row<KT, KLO>(w, e0[u] >= 0, sm + kOffK + kb * kTileBytes, r, sm + kOffK + kTileBytes);
                }
                tc::fence_proxy_async_smem();
                tc::mbar_arrive(bar(B_KFULL + kb));
                if (!__all_sync(0xffffffffu, j < 2 || wait(B_VEMPTY + b, ((j >> 1) - 1) & 1))) break;
#pragma unroll
                for (int u = 0; u < RPT; ++u) {
                    const int r = r0 + u * NPT;
                    uint32_t w[QSeg<VT>::NW];
#pragma unroll
                    for (int i = 0; i < QSeg<VT>::NW; ++i) w[i] = *reinterpret_cast<const uint32_t *>(raw_v(slot, r) + 4 * i);
                    store_row<VT>(w, e0[u] >= 0, sm + kOffV + b * kTileBytes, r);
                }
                tc::fence_proxy_async_smem();
                tc::mbar_arrive(bar(B_VFULL + b));
#pragma unroll
                for (int u = 0; u < RPT; ++u) {
                    e0[u] = e1[u];
                    e1[u] = e2[u];
                }
            }
            cp_async_wait<0>();
        }
    } else if (warp == C::kMmaWarp || warp == C::kPvWarp) {
        // ---------------- MMA issue -------------------------------------------
        // MODE 0: this warp's thread issues the S MMAs and the next warp's the
        // PV MMAs, so that PV of one tile and S of a later one go out side by
        // side (a thread's issue of eight MMAs takes about as long as the
        // tensor core runs them).  MODE 1 and 2: one thread issues S of tile
        // jj, then PV of tile jj-1.  Each issuer drains its own MMAs on abort:
        // a commit covers every MMA its thread issued before it.
        if (lane == 0 && n_tiles > 0) {
            // operand descriptors of the first K and V slots; the rest are offsets
            const uint64_t dk0 = tc::smem_desc(sbase + kOffK, 16, 1024);
            const uint64_t dv0 = tc::smem_desc(sbase + kOffV, kHalfTile, 1024);
            const uint64_t dq0 = tc::smem_desc(sbase + kOffQ, 16, 1024);   // Q (TMA instance)
            int last_bar = -1;                      // barrier and phase of this thread's last commit
            uint32_t last_par = 0;
            if constexpr (C::kSplitIssue) {
                if (warp == C::kMmaWarp) {
                    bool ok = wait(B_QFULL, 0);
                    tc::tc_fence_after();
                    for (int jj = 0; ok && jj < n_tiles; ++jj) {
                        const int b = jj & 1;
                        const int kb = KLO ? 0 : b;
                        const int sb = jj % kSBuf;
                        if (!wait(B_KFULL + kb, KLO ? (jj & 1) : ((jj >> 1) & 1))) break;
                        if (jj >= kSBuf && !wait(B_SFREE + sb, ((jj / kSBuf) - 1) & 1)) break;
                        tc::tc_fence_after();
                        const uint32_t d_s = tmem + static_cast<uint32_t>(sb * kPN);
                        constexpr int KSTEPS = (KLO ? 2 : 1) * kPD / 16;   // hi then lo
#pragma unroll
                        for (int ks = 0; ks < KSTEPS; ++ks) {
                            const int kk = ks % (kPD / 16);
                            const uint32_t off = (kk >> 2) * kHalfTile + (kk & 3) * 32;
                            const uint64_t bd = tc::desc_add(dk0, (KLO ? (ks / (kPD / 16)) : b) * kTileBytes + off);
                            if constexpr (P2)
                                tc::mma_f16_ss(d_s, tc::desc_add(dq0, off), bd, kIdescS, ks > 0);
                            else
                                tc::mma_f16_ts(d_s, tmem + static_cast<uint32_t>(kQCol + kk * 8), bd, kIdescS, ks > 0);
                        }
                        tc::mma_commit(bar(B_SFULL + sb));
                        tc::mma_commit(bar(B_KEMPTY + kb));
                        last_bar = B_SFULL + sb;
                        last_par = (jj / kSBuf) & 1;
                    }
                } else {
                    for (int j = 0; j < n_tiles; ++j) {
                        const int b = j & 1;
                        const int pb = P2 ? (j & 1) : 0;             // P buffer of tile j
                        if (!wait(B_PFULL + pb, (P2 ? (j >> 1) : j) & 1)) break;
                        if (!wait(B_VFULL + b, (j >> 1) & 1)) break;
                        tc::tc_fence_after();
                        const uint32_t d_o = tmem + kOCol;
#pragma unroll
                        for (int kk = 0; kk < kPN / 16; ++kk) {
                            // P of keys 16kk .. 16kk+15: fp16 pairs in columns kPCol + 8kk ..
                            const uint32_t a_t = tmem + static_cast<uint32_t>(kPCol + pb * (kPN / 2) + kk * 8);
                            // V tile as B in MN-major layout: 16 keys = 2048 bytes per k-step;
                            // the second 64-wide d block is kHalfTile away (leading offset),
                            // 8-key row groups are 1024 bytes apart (stride offset).
                            const uint64_t bd = tc::desc_add(dv0, b * kTileBytes + kk * 2048);
                            tc::mma_f16_ts(d_o, a_t, bd, kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
                        }
                        tc::mma_commit(bar(B_VEMPTY + b));
                        tc::mma_commit(bar(B_PFREE + pb));
                        last_bar = B_PFREE + pb;
                        last_par = (P2 ? (j >> 1) : j) & 1;
                    }
                }
            } else {
                bool ok = wait(B_QFULL, 0);
                tc::tc_fence_after();
                for (int jj = 0; ok && jj <= n_tiles; ++jj) {
                    if (jj < n_tiles) {
                        const int b = jj & 1;
                        const int kb = KLO ? 0 : b;
                        const int sb = jj % kSBuf;
                        if (!wait(B_KFULL + kb, KLO ? (jj & 1) : ((jj >> 1) & 1))) break;
                        if (jj >= kSBuf && !wait(B_SFREE + sb, ((jj / kSBuf) - 1) & 1)) break;
                        tc::tc_fence_after();
                        const uint32_t d_s = tmem + static_cast<uint32_t>(sb * kPN);
                        constexpr int KSTEPS = (KLO ? 2 : 1) * kPD / 16;   // hi then lo
#pragma unroll
                        for (int ks = 0; ks < KSTEPS; ++ks) {
                            const int kk = ks % (kPD / 16);
                            const uint32_t off = (kk >> 2) * kHalfTile + (kk & 3) * 32;
                            const uint64_t bd = tc::desc_add(dk0, (KLO ? (ks / (kPD / 16)) : b) * kTileBytes + off);
                            if constexpr (P2)
                                tc::mma_f16_ss(d_s, tc::desc_add(dq0, off), bd, kIdescS, ks > 0);
                            else
                                tc::mma_f16_ts(d_s, tmem + static_cast<uint32_t>(kQCol + kk * 8), bd, kIdescS, ks > 0);
                        }
                        tc::mma_commit(bar(B_SFULL + sb));
                        tc::mma_commit(bar(B_KEMPTY + kb));
                        last_bar = B_SFULL + sb;
                        last_par = (jj / kSBuf) & 1;
                    }
                    if (jj >= 1) {
                        const int j = jj - 1;
                        const int b = j & 1;
                        const int pb = P2 ? (j & 1) : 0;             // P buffer of tile j
                        if (!wait(B_PFULL + pb, (P2 ? (j >> 1) : j) & 1)) break;
                        if (!wait(B_VFULL + b, (j >> 1) & 1)) break;
                        tc::tc_fence_after();
                        const uint32_t d_o = tmem + kOCol;
#pragma unroll
                        for (int kk = 0; kk < kPN / 16; ++kk) {
                            // P of keys 16kk .. 16kk+15: fp16 pairs in columns kPCol + 8kk ..
                            const uint32_t a_t = tmem + static_cast<uint32_t>(kPCol + pb * (kPN / 2) + kk * 8);
                            // V tile as B in MN-major layout: 16 keys = 2048 bytes per k-step;
                            // the second 64-wide d block is kHalfTile away (leading offset),
                            // 8-key row groups are 1024 bytes apart (stride offset).
                            const uint64_t bd = tc::desc_add(dv0, b * kTileBytes + kk * 2048);
                            tc::mma_f16_ts(d_o, a_t, bd, kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
                        }
                        tc::mma_commit(bar(B_VEMPTY + b));
                        tc::mma_commit(bar(B_PFREE + pb));
                        last_bar = B_PFREE + pb;
                        last_par = (P2 ? (j >> 1) : j) & 1;
                    }
                }
            }
            if (*reinterpret_cast<volatile int *>(&s_abort) && last_bar >= 0)
                tc::mbar_wait(bar(last_bar), last_par, nullptr, 100000000ull);
        }
    } else {
        // ---------------- softmax warps (two threads per query row) -----------
        const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        // Q: this thread's half of its row (dims hf*64 ..) -> shared memory in
        // the swizzled K-major layout of a K tile (TMA instance), or tensor
        // memory columns kQCol + hf*32 .., two fp16 per column.
        {
            const __half *qp = a.q + ((static_cast<int64_t>(s) * a.nq + (row_ok ? t_row : 0)) * a.H + kh * a.G +
                                      (m % a.G)) * kPD + hf * 64;
            uint32_t qw[32];
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) {
                const uint4 v = row_ok ? *reinterpret_cast<const uint4 *>(qp + cc * 8) : make_uint4(0, 0, 0, 0);
                if constexpr (P2) {
                    *reinterpret_cast<uint4 *>(sm + kOffQ + tile_off(m, hf * 8 + cc)) = v;
                } else {
                    qw[4 * cc] = v.x;
                    qw[4 * cc + 1] = v.y;
                    qw[4 * cc + 2] = v.z;
                    qw[4 * cc + 3] = v.w;
                }
            }
            if constexpr (P2) {
                tc::fence_proxy_async_smem();
            } else {
                tc::tmem_st32u(lane_base + kQCol + hf * 32, qw);
                tc::tmem_wait_st();
                tc::tc_fence_before();
            }
            tc::mbar_arrive(bar(B_QFULL));
        }
        constexpr int NC = kPN / 2;                 // columns per thread
        // No early exit from this loop: the two warps of a row pair meet on a
        // named barrier every tile, so both must run every iteration.  After
        // a wait gives up, every later wait returns at once and the CTA runs
        // through to its exit (its outputs are then invalid and the status
        // word says so).
        for (int j = 0; j < n_tiles; ++j) {
            const int b = j & 1;                        // slot of the row-maximum exchange
            const int sb = j % kSBuf;                   // S buffer of this tile
            const int64_t key0 = j_lo + static_cast<int64_t>(j) * kPN + hf * NC;   // local index of column 0
            __all_sync(0xffffffffu, wait(B_SFULL + sb, (j / kSBuf) & 1));
            // Padding entries of a row list: one bit per column of this half,
            // published by the producers (entries past the split count as
            // present; lim_end masks them).
            uint32_t vm0 = 0xffffffffu, vm1 = 0xffffffffu;
            if (lrow) {
                __all_sync(0xffffffffu, wait(B_MFULL + (j & 3), (j >> 2) & 1));
                vm0 = s_vmask[j & 3][hf * 2];
                vm1 = s_vmask[j & 3][hf * 2 + 1];
            }
            tc::tc_fence_after();
            const int64_t pos0 = a.key_pos0 + a.logical0 + key0;
            const int64_t lim_pos = static_cast<int64_t>(pos_row) - pos0;   // columns > lim_pos are masked
            const int64_t lim_end = j_hi - key0;                            // columns >= lim_end are outside the split
            // This half's scores, masked only where a tile reaches past a
            // row's position or the split's end, or holds padding
            // (warp-uniform test; most tiles skip it).
            float x[NC];
            auto load_scores = [&](bool release) {
                uint32_t sr[NC / 32][32];
#pragma unroll
                for (int c = 0; c < NC / 32; ++c) tc::tmem_ld32(lane_base + sb * kPN + hf * NC + c * 32, sr[c]);
#pragma unroll
                for (int c = 0; c < NC / 32; ++c) tc::tmem_wait_ld(sr[c]);
                if (release) {
                    tc::tc_fence_before();
                    tc::mbar_arrive(bar(B_SFREE + sb));   // the S buffer may take the next tile's S
                }
#pragma unroll
                for (int c = 0; c < NC / 32; ++c)
#pragma unroll
                    for (int i = 0; i < 32; ++i) x[c * 32 + i] = __uint_as_float(sr[c][i]);
                if (__any_sync(0xffffffffu, lim_pos < NC - 1 || lim_end < NC || (vm0 & vm1) != 0xffffffffu)) {
#pragma unroll
                    for (int i = 0; i < NC; ++i) {
                        const bool present = ((i < 32 ? vm0 : vm1) >> (i & 31)) & 1u;
                        if (i > lim_pos || i >= lim_end || !present) x[i] = -INFINITY;
                    }
                }
            };
            load_scores(!P2);
            if (P2 && j > 0) {
                // the previous tile's P store has landed by now: publish it
                // (its PV is not urgent with two P buffers)
                tc::tmem_wait_st();
                tc::tc_fence_before();
                tc::mbar_arrive(bar(B_PFULL + ((j - 1) & 1)));
            }
            // Row maximum on the raw scores (the scale is positive): this
            // half's four chains, then the partner half's value.
            float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int i = 0; i < NC; i += 4) {
                mq[0] = fmaxf(mq[0], x[i]);
                mq[1] = fmaxf(mq[1], x[i + 1]);
                mq[2] = fmaxf(mq[2], x[i + 2]);
                mq[3] = fmaxf(mq[3], x[i + 3]);
            }
            const float mh = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
            s_pair[b][hf][m] = mh;
            // p = 2^(s * scale_log2 - ref): one FMA and one exp2 per score.
            float ls[4];
            uint32_t ph[NC / 2];
            auto exps = [&](float nref) {
#pragma unroll
                for (int q = 0; q < 4; ++q) ls[q] = 0.f;
#pragma unroll
                for (int i = 0; i < NC; i += 2) {
                    const float p0 = fast_exp2(fmaf(x[i], a.scale_log2, nref));
                    const float p1 = fast_exp2(fmaf(x[i + 1], a.scale_log2, nref));
                    ls[(i >> 1) & 3] += p0 + p1;
                    ph[i / 2] = pack_half2(p0, p1);
                }
            };
            // TMA instance: the exponentials are first taken against the
            // current reference, which stays unless the row maximum grew by
            // more than 2^8 (rare after a row's first tile), while the partner
            // half is still on its way to the exchange; a warp with a row
            // whose reference moves loads its scores again and takes them over,
            // and the S buffer is released once that is settled (the S MMAs
            // run ahead).  The software-producer instances, at 128 registers,
            // exchange first and keep no second pass.
            if constexpr (P2) exps(m_ref == -INFINITY ? 0.f : -m_ref);
            pair_sync();
            const float mx = fmaxf(mh, s_pair[b][hf ^ 1][m]) * a.scale_log2;
            const float m_new = fmaxf(m_ref, mx);
            const bool resc = m_new > m_ref + kRescaleLog2;   // true on the first finite maximum
            const float ref = resc ? m_new : m_ref;
            const float alpha = resc ? fast_exp2(m_ref - ref) : 1.f;
            if constexpr (P2) {
                if (__any_sync(0xffffffffu, resc)) {
                    load_scores(false);
                    exps(ref == -INFINITY ? 0.f : -ref);
                }
                tc::tc_fence_before();
                tc::mbar_arrive(bar(B_SFREE + sb));       // the S buffer may take the next tile's S
            } else {
                exps(ref == -INFINITY ? 0.f : -ref);
            }
            l_run = l_run * alpha + ((ls[0] + ls[1]) + (ls[2] + ls[3]));   // this half's columns
            m_ref = ref;
            // P's buffer is free once PV of the tile before last (two P
            // buffers) or of the previous tile (one) is done.  O is rescaled
            // only when the reference maximum moved (rarely), once PV of the
            // previous tile is done.
            const int pb = P2 ? (j & 1) : 0;
            if (j >= (P2 ? 2 : 1)) {
                __all_sync(0xffffffffu, wait(B_PFREE + pb, (P2 ? (j >> 1) - 1 : j - 1) & 1));
                tc::tc_fence_after();
            }
            const bool resc_o = j > 0 && __any_sync(0xffffffffu, alpha != 1.f);
            if (P2 && resc_o) {
                __all_sync(0xffffffffu, wait(B_PFREE + ((j - 1) & 1), ((j - 1) >> 1) & 1));
                tc::tc_fence_after();
            }
            if (resc_o) {
#pragma unroll
                for (int c = 0; c < NC / 32; ++c) {
                    uint32_t rr[32];
                    tc::tmem_ld32(lane_base + kOCol + hf * NC + c * 32, rr);
                    tc::tmem_wait_ld(rr);
                    float v[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(rr[i]) * alpha;
                    tc::tmem_st32(lane_base + kOCol + hf * NC + c * 32, v);
                }
            }
            // P (fp16 pairs): keys hf*64 + 2c, +1 in column kPCol + 64 pb + hf*32 + c;
            // the TMA instance publishes it after the next tile's scores are
            // loaded, so that the store lands under that load
            tc::tmem_st32u(lane_base + kPCol + pb * (kPN / 2) + hf * (NC / 2), ph);
            if constexpr (!P2) {
                tc::tmem_wait_st();
                tc::tc_fence_before();
                tc::mbar_arrive(bar(B_PFULL + pb));
            }
        }
        if (P2 && n_tiles > 0) {
            tc::tmem_wait_st();
            tc::tc_fence_before();
            tc::mbar_arrive(bar(B_PFULL + ((n_tiles - 1) & 1)));
        }
        // ---------------- epilogue: O / l, lse -------------------------------
        float ov[NC];
        bool have = n_tiles > 0 && !*reinterpret_cast<volatile int *>(&s_abort);
        if (have) {                                            // the last PV
            const int jl = n_tiles - 1;
            have = wait(B_PFREE + (P2 ? (jl & 1) : 0), (P2 ? (jl >> 1) : jl) & 1);
        }
        have = __all_sync(0xffffffffu, have);
        if (have) {
            tc::tc_fence_after();
            uint32_t orr[NC / 32][32];
#pragma unroll
            for (int c = 0; c < NC / 32; ++c) tc::tmem_ld32(lane_base + kOCol + hf * NC + c * 32, orr[c]);
#pragma unroll
            for (int c = 0; c < NC / 32; ++c) tc::tmem_wait_ld(orr[c]);
#pragma unroll
            for (int c = 0; c < NC / 32; ++c)
#pragma unroll
                for (int i = 0; i < 32; ++i) ov[c * 32 + i] = __uint_as_float(orr[c][i]);
        }
        // the row's sum is the two halves' sums
        s_pair[2][hf][m] = l_run;
        pair_sync();
        const float l_row = l_run + s_pair[2][hf ^ 1][m];
        if (row_ok) {
            const int64_t r = (static_cast<int64_t>(s) * a.nq + t_row) * a.H + kh * a.G + (m % a.G);
            const bool direct = a.n_splits == 1;
            float *op = (direct ? a.o_out + r * kPD : a.o_split + (static_cast<int64_t>(split) * a.R + r) * kPD) +
                        hf * NC;
            float *lp = direct ? a.lse_out + r : a.lse_split + static_cast<int64_t>(split) * a.R + r;
            if (!have || m_ref == -INFINITY || l_row <= 0.f) {
#pragma unroll
                for (int i = 0; i < NC; i += 4) *reinterpret_cast<float4 *>(op + i) = make_float4(0.f, 0.f, 0.f, 0.f);
                if (hf == 0) *lp = -INFINITY;
            } else {
                const float inv = 1.f / l_row;
#pragma unroll
                for (int i = 0; i < NC; i += 4)
                    *reinterpret_cast<float4 *>(op + i) =
                        make_float4(ov[i] * inv, ov[i + 1] * inv, ov[i + 2] * inv, ov[i + 3] * inv);
                if (hf == 0) *lp = (m_ref + __log2f(l_row)) * 0.6931471805599453f;
            }
        }
    }

    // ---------------- teardown, then the cross-split merge --------------------
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc::tc_fence_after();
        tc::tmem_dealloc<512>(tmem);
    }
    if (a.n_splits == 1) return;
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = atomicAdd(a.counters + unit, 1) == a.n_splits - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (row_ok) {
        // thread (row, half) merges its 64 columns over the splits
        const int64_t r = (static_cast<int64_t>(s) * a.nq + t_row) * a.H + kh * a.G + (m % a.G);
        float M = -INFINITY;
        for (int sp = 0; sp < a.n_splits; ++sp) M = fmaxf(M, __ldcg(a.lse_split + static_cast<int64_t>(sp) * a.R + r));
        float *op = a.o_out + r * kPD + hf * 64;
        if (M == -INFINITY) {
            for (int i = 0; i < 64; i += 4) *reinterpret_cast<float4 *>(op + i) = make_float4(0.f, 0.f, 0.f, 0.f);
            if (hf == 0) a.lse_out[r] = -INFINITY;
        } else {
            float acc[64];
#pragma unroll
            for (int i = 0; i < 64; ++i) acc[i] = 0.f;
            float W = 0.f;
            for (int sp = 0; sp < a.n_splits; ++sp) {
                const float l = __ldcg(a.lse_split + static_cast<int64_t>(sp) * a.R + r);
                if (l == -INFINITY) continue;
                const float w = fast_exp2((l - M) * 1.4426950408889634f);
                W += w;
                const float4 *src = reinterpret_cast<const float4 *>(
                    a.o_split + (static_cast<int64_t>(sp) * a.R + r) * kPD + hf * 64);
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float4 v = __ldcg(src + i);
                    acc[4 * i] = fmaf(w, v.x, acc[4 * i]);
                    acc[4 * i + 1] = fmaf(w, v.y, acc[4 * i + 1]);
                    acc[4 * i + 2] = fmaf(w, v.z, acc[4 * i + 2]);
                    acc[4 * i + 3] = fmaf(w, v.w, acc[4 * i + 3]);
                }
            }
            const float inv = 1.f / W;
            for (int i = 0; i < 64; i += 4)
                *reinterpret_cast<float4 *>(op + i) = make_float4(acc[i] * inv, acc[i + 1] * inv, acc[i + 2] * inv,
                                                                  acc[i + 3] * inv);
            if (hf == 0) a.lse_out[r] = M + __logf(W);
        }
    }
    if (tid == 0) a.counters[unit] = 0;
}

namespace {
// One cache per instance and translation unit (internal linkage, see
// decode_attr_cache).
template <int MODE, int KT, int VT>
KernelAttrCache &prefill_attr_cache()
{
    static KernelAttrCache c;
    return c;
}
}  // namespace

// Launch one instance (its shared-memory opt-in is made once per device).
template <int MODE, int KT, int VT>
int launch_prefill_t(skv_handle *h, const CUtensorMap &mk, const CUtensorMap &mv, const PrefillArgs &a, dim3 grid,
                     cudaStream_t st)
{
    cudaError_t e = kernel_smem_optin(prefill_attr_cache<MODE, KT, VT>(), reinterpret_cast<const void *>(splitkv_prefill_kernel<MODE, KT, VT>),
                                      smem_bytes<MODE, KT, VT>(), Cfg<MODE>::kThreads, nullptr);
    if (e != cudaSuccess) return cuda_fail(h, e, "cudaFuncSetAttribute(prefill)");
    if (h->prof_before) cudaEventRecord(h->prof_before, st);
    splitkv_prefill_kernel<MODE, KT, VT><<<grid, Cfg<MODE>::kThreads, smem_bytes<MODE, KT, VT>(), st>>>(mk, mv, a);
    if (h->prof_after) cudaEventRecord(h->prof_after, st);
    return cuda_fail(h, cudaGetLastError(), "prefill kernel launch");
}

// Software-producer instances (prefill_sw.cu).
int launch_prefill_sw(skv_handle *h, const PrefillArgs &a, int kt, int vt, dim3 grid, cudaStream_t st);
// Two query tiles per CTA over dense q8_0 / q4_0 keys and q4_0 values
// (prefill_pairq.cu); grid x = (KV head, query-tile pair).
int launch_prefill_pairq(skv_handle *h, const PrefillArgs &a, int kt, dim3 grid, cudaStream_t st);

}  // namespace pf
}  // namespace skv
