// Device-side data layout shared by the host library and the kernels.
//
// A step streams two tables, both built on the host from the caller's list
// and uploaded once per distinct list:
//
//   * the update table covers every trainable element; the norm table covers
//     the trainable, owned elements only (non-owned entries never reach the
//     square-sum kernel, so that kernel has no ownership branch);
//   * a table is a sequence of segments -- a contiguous element range of one
//     tensor -- grouped into chunks of about the same number of elements.
//     One CTA processes one chunk at a time.  Small tensors share a chunk,
//     large tensors are cut into several; so one launch covers the whole
//     list however many tensors it has (the case of many small tensors that
//     the SomaSpeed optimizer paragraphs single out).
//
// Vector body: inside a segment, elements [head, head + 8*nvec) are processed
// eight at a time with 16-byte accesses, or 32-byte ones for fp32 buffers
// that are 32-byte aligned there; the host picks `head` so that every buffer
// is 16-byte aligned there (32-byte for fp32 ones when possible), and cuts
// tensors only at such points.  The few elements before and after run one at
// a time.  A tensor whose buffers cannot all be aligned at one element is
// processed one element at a time.
#pragma once

#include <cmath>
#include <cstdint>

namespace soma {

constexpr int kVec = 8;                 // elements per vector step
constexpr int kMaxSegsPerChunk = 64;    // bounds the shared-memory segment cache
constexpr int kMaxGroups = 64;

enum : int32_t { kNone = 0, kF32 = 0, kBF16 = 1, kF16 = 2 };

struct Seg {                // 64 bytes
    float* p;               // already offset to the segment's first element
    const void* g;
    float* m;
    float* v;
    void* plow;             // bf16/fp16 copy of p written by the update, or nullptr
    int32_t len;            // elements in the segment
    int32_t head;           // scalar elements before the vector body
    int32_t nvec;           // 8-element vectors in the body
    uint16_t group;
    uint8_t gdtype;         // kF32, kBF16, kF16
    uint8_t lowdt;          // kNone, kBF16, kF16
    uint64_t pad;
};
static_assert(sizeof(Seg) == 64, "Seg layout");

// Per-group constants of one step, derived in fp64 and rounded once to fp32.
struct GroupHp {
    float decay;            // 1 - lr * weight_decay
    float beta1, one_minus_beta1;
    float beta2, one_minus_beta2;
    float step_size;        // lr / (1 - beta1^t)
    float inv_sqrt_bc2;     // 1 / sqrt(1 - beta2^t)
    float eps;
};

// fp64 operations rounded to nearest one at a time (never fused into an
// FMA), so that the host, for regular steps, and the device, for graph
// steps, derive the same constants bit for bit.
#if defined(__CUDA_ARCH__)
#define SOMA_HD __host__ __device__
#define SOMA_DMUL(a, b) __dmul_rn(a, b)
#define SOMA_DSUB(a, b) __dsub_rn(a, b)
#define SOMA_DDIV(a, b) __ddiv_rn(a, b)
#define SOMA_DSQRT(a) __dsqrt_rn(a)
#elif defined(__CUDACC__)
#define SOMA_HD __host__ __device__
#define SOMA_DMUL(a, b) ((a) * (b))
#define SOMA_DSUB(a, b) ((a) - (b))
#define SOMA_DDIV(a, b) ((a) / (b))
#define SOMA_DSQRT(a) sqrt(a)
#else
#define SOMA_HD
#define SOMA_DMUL(a, b) ((a) * (b))
#define SOMA_DSUB(a, b) ((a) - (b))
#define SOMA_DDIV(a, b) ((a) / (b))
#define SOMA_DSQRT(a) sqrt(a)
#endif

// b^t for an integer t >= 0 by repeated squaring: at most 2 log2(t) + 1
// multiplies (fp64 transcendental functions are slow on this GPU).
SOMA_HD inline double pow_step(double b, int64_t t) {
    double r = 1.0;
    while (t > 0) {
        if (t & 1) r = SOMA_DMUL(r, b);
        b = SOMA_DMUL(b, b);
        t >>= 1;
    }
    return r;
}

// Constants of a group at step t (bias corrections 1 - beta^t of AdamW).
SOMA_HD inline GroupHp make_group_hp(double lr, double beta1, double beta2, double eps, double weight_decay,
                                     int64_t t) {
    const double bc1 = SOMA_DSUB(1.0, pow_step(beta1, t));
    const double bc2 = SOMA_DSUB(1.0, pow_step(beta2, t));
    GroupHp h;
    h.decay = (float)SOMA_DSUB(1.0, SOMA_DMUL(lr, weight_decay));
    h.beta1 = (float)beta1;
    h.one_minus_beta1 = (float)SOMA_DSUB(1.0, beta1);
    h.beta2 = (float)beta2;
    h.one_minus_beta2 = (float)SOMA_DSUB(1.0, beta2);
    h.step_size = (float)SOMA_DDIV(lr, bc1);
    h.inv_sqrt_bc2 = (float)SOMA_DDIV(1.0, SOMA_DSQRT(bc2));
    h.eps = (float)eps;
    return h;
}

// Written by the square-sum kernel's last CTA, read by the update kernel and
// by soma_opt_get_norm.
struct Result {
    double sumsq;           // sum over owned elements of g^2, or of (g / d_group)^2 with group divisors
    double norm;            // the global norm of the normalized gradients
    double coef;            // min(1, max_norm / (norm + 1e-6))
    float scale;            // coef / d in fp32: the update multiplies g by this
    uint32_t nonfinite;     // 1 when norm is not finite
    uint32_t ticket;        // CTA arrival counter; the last CTA resets it to 0
    uint32_t nonfinite_steps;  // steps with a non-finite norm since the host last cleared it
    uint32_t pad[2];
};
static_assert(sizeof(Result) == 48, "Result layout");

// Device copy of a group's hyperparameters and step count, used by the
// graph-capturable step (the layout of soma_device_group_t in soma_opt.h).
struct DevGroup {           // 64 bytes
    double lr, beta1, beta2, eps, weight_decay;
    int64_t step;
    int64_t reserved[2];
};
static_assert(sizeof(DevGroup) == 64, "DevGroup layout");

struct Table {
    const Seg* segs;
    const int32_t* chunk_begin;  // nchunks + 1 entries
    int32_t nchunks;
};

struct NormArgs {
    Table t;
    double* partials;       // one per chunk
    Result* res;
    double divisor;         // the step's divisor d
    double inv_step_divisor;  // 1 / d, rounded once (fp64 division is slow on the device)
    double max_norm;
    double inv_divisor[kMaxGroups];  // 1 / (effective divisor) of each group
    // group divisors only: the last CTA writes c / d of each group here
    float* gscale;
    // graph-capturable step only: CTA 0 (launched in addition to the chunk
    // CTAs) advances the step count of every group whose bit is set in
    // `present` and writes its constants
    DevGroup* dgroups;
    GroupHp* dhp;
    uint64_t present;
    int32_t ngroups;
    // multi-rank step: when set, the last CTA also stores this rank's
    // normalized square-sum S / d^2 here
    double* sumsq_out;
};

// Multi-rank step: one thread adds the ranks' normalized square-sums in rank
// order and derives norm, c and the update scale.
struct FinishArgs {
    const double* parts;
    int32_t count;
    Result* res;
    double divisor;
    double inv_step_divisor;
    double max_norm;
    // group divisors only: gscale[q] = c / d_q for q < ngroups
    float* gscale;
    int32_t ngroups;
    double inv_divisor[kMaxGroups];
};

struct UpdateArgs {
    Table t;
    const Result* res;
    GroupHp groups[kMaxGroups];   // regular step: constants as kernel arguments
    const GroupHp* dhp;           // graph-capturable step: constants in device memory
    int32_t ngroups;
    const float* gscale;          // group divisors: c / d of each group, written by the norm side
};

// Host-side cutting rule shared by every table builder.  A segment that
// starts at element `off` of an n-element tensor with vector head h (-1 =
// no vector body) and may take up to `room` elements ends at the returned
// element: a cut inside the tensor is moved up to the vector grid h + 8j, so
// that only a tensor's first and last segments have scalar elements outside
// their vector bodies.
inline int64_t segment_cut(int64_t off, int64_t n, int64_t room, int h) {
    int64_t cut = off + (n - off < room ? n - off : room);
    if (h >= 0 && cut < n && cut > h) {
        cut = h + (cut - h + kVec - 1) / kVec * kVec;
        if (cut > n) cut = n;
    }
    return cut;
}

// head and nvec of the segment [off, off + len) of a tensor with vector head h.
inline void segment_body(int64_t off, int64_t len, int h, Seg& s) {
    s.len = (int32_t)len;
    if (h < 0) {
        s.head = (int32_t)len;
        s.nvec = 0;
    } else {
        s.head = off < h ? (int32_t)(h - off < len ? h - off : len) : 0;
        s.nvec = (int32_t)((len - s.head) / kVec);
    }
}

constexpr int kNormBlock = 512;
constexpr int kUpdateBlock = 256;

// Launch wrappers (kernels.cu).  Return the cudaError_t of the launch as int.
// graph = true selects the variants that take group constants from device
// memory (NormArgs::dgroups / dhp, UpdateArgs::dhp).
// group_div: some group of the list sets its own divisor (NormArgs::inv_divisor).
// overlap (here and for launch_update) = true launches with programmatic
// stream serialization: the kernel may start while the previous kernel on the
// stream finishes, and waits (griddepcontrol.wait) before it reads anything
// that kernel may write.  The update kernel lets the next square-sum kernel
// start this way, and the square-sum kernel the update kernel.
int launch_norm(const NormArgs& a, int grid, void* stream, bool graph = false, bool group_div = false,
                bool overlap = false);
int launch_update(const UpdateArgs& a, int grid, void* stream, bool graph = false, bool overlap = false,
                  bool group_div = false);
int launch_finish(const FinishArgs& a, void* stream);

// Single-launch step (small lists): one cluster of `ctas` CTAs does the
// square-sum, the norm and the update.  `ctas` must be a value
// small_step_cluster_size() returned.  overlap as above; graph = true takes
// the group constants from NormArgs::dgroups and advances the step counts
// there (UpdateArgs::groups unused); group_div as for launch_norm.
constexpr int kSmallStepMaxCtas = 16;
int small_step_cluster_size();  // largest cluster (16, 8, 4, 2) the device can run, else 0
int launch_small_step(const NormArgs& na, const UpdateArgs& ua, int ctas, void* stream, bool overlap = false,
                      bool graph = false, bool group_div = false);

}  // namespace soma
