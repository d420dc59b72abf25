// Internal interface between the C ABI (abi.cpp) and the kernels
// (kernels.cu): launch arguments, plans and the shared-memory layout, which
// the host sizes and the device carves up with the same function.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace cs {

// Consumer warps per CTA of the streaming kernels. Two more warps issue the
// bulk copies: kConsumerWarps lanes of one warp the candidate stages (lane l
// fills exactly the ring slots consumer warp l drains), one lane of the
// other the query rows.
constexpr int kConsumerWarps = 8;
constexpr int kStreamThreads = (kConsumerWarps + 2) * 32;
// On-chip per-row results per question (K <= 255), one buffer per question
// in flight.
constexpr int kLogitSlots = 256;
// Most candidate rows in one ring stage; one warp reduces a whole stage.
constexpr int kMaxRowsPerStage = 8;
// Plans whose stages hold at most this many rows run a short-stage build of
// the fused kernels (less code to fetch on a batch-1 launch).
constexpr int kSmallStageRows = 2;
// Largest cluster the split plan uses (non-portable size on sm_100-class parts).
constexpr int kMaxCluster = 16;
// Threads of the scalar fallback kernel.
constexpr int kGenericThreads = 256;

// The float32 arguments of one readout, after validation.
struct Problem {
    const float* Q;    // [B][D]
    const void* C;     // [B][K][D], float32 or bfloat16 (see c_bf16)
    float* out;        // [B][K]
    long long B;
    int K;
    int D;
    int normalize;     // 1 cosine, 0 dot
    // The logit factor a = scale / temperature, split by the host (which
    // forms it in double precision and refuses |a| > 2^126) into the signed
    // value scale w0 and the exponent scale kexp = |a| log2(e) / |w0| of
    // softmax_form.cuh: w0 = sign(a) for the cosine, and for the dot sign(a)
    // or, when |a| < 2^-100, sign(a) / 2.
    float w0;
    float kexp;
    float* staged;     // unfused baseline only: one float per row [B][K]
    int c_bf16;        // 1: C holds bfloat16 bit patterns (2 bytes each)
    // Ragged batches: question b owns rows offsets[b] .. offsets[b+1]-1 of C
    // (and of out); offsets has B+1 entries and total_rows = offsets[B].
    // nullptr: every question has K rows (row b*K + k).
    const long long* offsets;
    long long total_rows;
};

// Bytes of one element of C.
inline int c_elem_bytes(const Problem& p) { return p.c_bf16 ? 2 : 4; }

enum PlanKind { kPlanAuto = 0, kPlanStream = 1, kPlanCluster = 2, kPlanGeneric = 3, kPlanDirect = 4 };
// DIRECT plan: at most this many rows of a question per CTA, q and rows
// loaded into registers (chunks per lane nq4 in {1, 2, 4}); the wide form
// (long rows: q in shared memory) takes kDirectWideChunks 16-byte chunks of
// a row per lane, at most kDirectWideMaxRows rows per CTA and D up to
// kDirectWideMaxD.
constexpr int kDirectMaxRows = 32;
constexpr int kDirectWideChunks = 20;
constexpr int kDirectWideMaxRows = 16;
constexpr int kDirectWideMaxD = 5120;

struct Plan {
    int kind;          // PlanKind
    int cluster;       // CTAs per cluster (split plan), else 1
    int ctas;          // CTAs launched in total
    int rows_per_stage;// candidate rows per bulk-copy stage
    int stages;        // stages in the shared-memory ring
    int nq4;           // 16-byte chunks of a C row per lane whose q sits in registers (0: q read from
                       // smem); negative for unaligned rows (kNqcUnaligned, unaligned_nqc)
    size_t smem;       // dynamic shared memory per CTA
};

// Shared-memory carve-up of the streaming kernels. All offsets are bytes
// from the (128-byte aligned) dynamic shared-memory base.
struct SmemLayout {
    size_t ring;        // stages slots of slot_bytes each
    size_t slot_bytes;  // one ring slot: rows_per_stage rows of C
    size_t qbuf;        // 2 slots of qslot_bytes: the query rows
    size_t qslot_bytes;
    size_t tn;          // 2 buffers x (dot[kLogitSlots], squared norm[kLogitSlots]) floats
    size_t xch;         // kMaxCluster float2 (max, sum) received from the cluster's CTAs
    size_t bars;        // full[stages], empty[stages], qfull[2], qempty[2], xbar (8 B each)
    size_t range;       // two long longs: this CTA's question range (ragged STREAM plan)
    size_t flag;        // int: this CTA gave up waiting
    size_t total;
};

// Bulk copies of rows that do not start on a 16-byte boundary (or whose
// length is not a multiple of 16 bytes) copy the 16-byte aligned span
// around them: up to 15 bytes before and after, within the same 16-byte
// granules as the rows' own bytes. A slot holds that span.
__host__ __device__ inline size_t span_bytes(size_t bytes) { return (bytes + 15) / 16 * 16 + 32; }

// c_bytes: bytes of one element of C (4 float32, 2 bfloat16). unaligned:
// slots sized for the aligned spans of rows at any 4-byte (float32) or
// 2-byte (bfloat16) offset.
__host__ __device__ inline SmemLayout smem_layout(int stages, int rows_per_stage, int D, int c_bytes,
                                                  bool unaligned = false) {
    SmemLayout L;
    size_t off = 0;
    const size_t stage = (size_t)rows_per_stage * D * c_bytes, q = (size_t)D * sizeof(float);
    L.slot_bytes = unaligned ? span_bytes(stage) : stage;
    L.qslot_bytes = unaligned ? span_bytes(q) : q;
    L.ring = off;   off += (size_t)stages * L.slot_bytes;
    L.qbuf = off;   off += 2 * L.qslot_bytes;
    L.tn = off;     off += 4 * (size_t)kLogitSlots * sizeof(float);
    L.xch = off;    off += (size_t)kMaxCluster * 8;
    L.bars = off;   off += (2 * (size_t)stages + 5) * 8;
    L.range = off;  off += 16;
    L.flag = off;   off += 16;
    L.total = off;
    return L;
}

// Plan.nq4 of the streaming kernels for rows the bulk copies take as
// aligned spans (D not a multiple of 16 bytes' worth of elements, or Q or C
// off a 16-byte boundary). kNqcUnaligned: scalar shared-memory reads, q in
// shared memory, any D. unaligned_nqc(NU) = -NU, NU in {4, 8, 16}: rows read
// in 4-byte units (one float32 element, or a pair of bfloat16 elements), NU
// units a lane with q for them in registers; the plan takes the smallest NU
// with 32 NU >= the row's units (D float32, floor(D / 2) bfloat16), so that
// for NU > 4 a lane's first NU / 2 units are always inside the row.
constexpr int kNqcUnaligned = -1;
constexpr int kUnalignedUnits[3] = {4, 8, 16};
__host__ __device__ constexpr int unaligned_nqc(int nu) { return -nu; }
__host__ __device__ constexpr int unaligned_units(int nqc) { return nqc < -1 ? -nqc : 0; }

// What one launch of the streaming kernel computes.
enum StreamMode {
    kFusedCos = 0,   // the fused readout, cosine
    kFusedDot = 1,   // the fused readout, dot
    kRowNorm = 2,    // unfused baseline pass 1 (cosine): staged[row] = |c|
    kRowDot = 3,     // unfused baseline pass 1 (dot):    staged[row] = c . q
    kStagedCos = 4,  // unfused baseline pass 2 (cosine): dots, norms read from staged, softmax
};

// Launchers (kernels.cu). Each enqueues exactly one kernel on `stream` and
// returns the launch status; none synchronizes or allocates.
cudaError_t launch_stream(const Problem& p, const Plan& plan, int mode, cudaStream_t stream);
// G = 1: one CTA per question; G > 1: each question over a cluster of G CTAs
// (uniform K, B <= 65535).
cudaError_t launch_generic(const Problem& p, int G, cudaStream_t stream);
int max_active_generic_clusters(int cluster, int normalize, int c_bf16);
// Unfused baseline pass 2 (dot): softmax of a * staged (a the logit factor).
cudaError_t launch_staged_softmax(const Problem& p, cudaStream_t stream);

// Size, in floats, of the built-in staged array of the no-allocation
// unfused entry point (4 MiB): it serves calls with B*K up to this many rows.
constexpr unsigned long long kNoAllocStagedFloats = 1ull << 20;
// Device address of that array on `device` (which must be current), looked
// up once per device with cudaGetSymbolAddress and then cached.
cudaError_t noalloc_staged_address(int device, float** ptr);

// One-time per-device kernel attributes (dynamic smem ceiling, cluster size).
cudaError_t configure_device_kernels(int smem_optin);

// Clusters of `cluster` CTAs with `smem` bytes each that fit on the device
// at once (0 if none).
int max_active_clusters(int cluster, size_t smem, int nq4, int normalize, int c_bf16, int rows_per_stage);
// DIRECT plan (fused modes only): grid (cluster, B), clusters of `cluster`
// CTAs when cluster > 1; B <= 65535.
cudaError_t launch_direct(const Problem& p, const Plan& plan, cudaStream_t stream);
int max_active_direct_clusters(int cluster, int nq4, int normalize, int c_bf16);

// Bounded-wait self-test: one wait that nothing completes, limit_ns long.
cudaError_t launch_selftest_wait(unsigned long long limit_ns, cudaStream_t stream);

// Projections on the tensor cores (project.cu). H, W: bfloat16 bit
// patterns, row-major [rows][Din] and [D][Din]; D in {256, 512}, Din a
// multiple of 64; 16-byte aligned pointers.
size_t proj_smem_bytes(int D);
cudaError_t configure_proj_kernels(int smem_optin);
cudaError_t launch_project_rows(const uint16_t* H, const uint16_t* W, long long rows, int Din, int D, float* P,
                                int sms, unsigned* status, unsigned* bounds, cudaStream_t stream);
cudaError_t launch_project_score(const uint16_t* Hc, const uint16_t* Wc, const float* qproj, int B, int K, int Din,
                                 int D, int normalize, float w0, float kexp, float* out, int sms, unsigned* status,
                                 unsigned* bounds, cudaStream_t stream);
// Device address of the status word on the current device (for kernels in
// other translation units).
cudaError_t status_word_address(unsigned** ptr);

// Bounds-checked builds (compiled with -DCS_DEBUG_BOUNDS; the tests use one
// in place of a memory checker): before every global-memory access of the
// kernels, the range is checked against the extent of its buffer; a failing
// check records its site number (BoundsSite) in the bounds word if that is
// still 0, sets kDevErrBounds in the status word and skips the access.
// Release builds compile the checks away.
constexpr unsigned kDevErrBounds = 8u;
// Device status bit: a question's dot products or squared norms left
// float32's range (or an input was not finite), so it was skipped unscored.
constexpr unsigned kDevErrRange = 16u;
enum BoundsSite : unsigned {
    kSiteCopyC = 1,        // stream producer: rows of C
    kSiteRing = 2,         // stream producer: the ring slot they land in
    kSiteCopyQ = 3,        // query producer: q
    kSiteQbuf = 4,         // query producer: the q slot
    kSiteOut = 5,          // softmax of a question (STREAM plan)
    kSiteOutCluster = 6,   // softmax rows of a CTA (CLUSTER plan)
    kSiteStagedWrite = 7,  // unfused pass 1
    kSiteStagedRead = 8,   // unfused pass 2 (cosine)
    kSiteOffsets = 9,      // ragged: a question's offsets
    kSiteOffsetsSearch = 10,  // ragged: the CTA's first and last question
    kSiteGenericC = 11,
    kSiteGenericQ = 12,
    kSiteGenericOut = 13,
    kSiteStagedSoftmax = 14,     // unfused pass 2 (dot): staged similarities
    kSiteStagedSoftmaxOut = 15,
    kSitePeer = 16,        // cluster exchange slot in a peer CTA
    kSitePrefetchC = 17,   // stream prologue: L2 prefetch of the first rows
    kSiteUnitSlot = 18,    // unaligned unit-wise reads: the stage's extent in its ring slot
    kSiteProjQ = 20,       // projected readout: projected query
    kSiteProjOut = 21,     // projected readout: probabilities
    kSiteProjRows = 22,    // projected rows: a 32-byte row segment of P
    kSiteSelftest = 99,
};
bool debug_bounds_build();
cudaError_t bounds_site_address(unsigned** ptr);
cudaError_t read_bounds_site(unsigned* site, bool clear);
// Bounds-checked builds: one thread checks an address one past a buffer's
// end (arithmetic only, nothing is accessed); cudaErrorNotSupported otherwise.
cudaError_t launch_selftest_bounds(cudaStream_t stream);

// Device status word (bounded-wait give-ups).
cudaError_t read_device_status(unsigned* flags, bool clear);

}  // namespace cs
