/*
 * ebin -- ONNX broadcast binary elementwise engine for one NVIDIA GB300 GPU.
 *
 * C ABI.  Plain pointers and sizes only; no C++ or PyTorch types.
 *
 * The engine follows the three-stage statement of "Binary Kernel Design"
 * (onnx-light-cpu), section "Prepared execution": a descriptor is built once
 * per node, a plan is built (or fetched from a bounded 8-entry LRU) once per
 * pair of concrete input shapes, and the plan is executed on device buffers.
 *
 * Threading: every entry point is thread-safe.  Descriptors and plans are
 * immutable after creation and may be shared between host threads and CUDA
 * streams.
 *
 * Streams: `stream` arguments are a cudaStream_t passed as void* (NULL = the
 * legacy default stream).  Kernels are enqueued; nothing synchronises unless
 * stated.
 *
 * Device pointers: A, B and out of ebin_execute are device (or managed)
 * memory on the current CUDA device, owned by the caller, laid out dense
 * row-major (C order) in the element type of the descriptor.
 */
#ifndef EBIN_H
#define EBIN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define EBIN_MAX_RANK 8
/* element counts and view extents stay below this (2^60) */
#define EBIN_MAX_ELEMENTS (((int64_t)1) << 60)
#define EBIN_PLAN_CACHE_CAPACITY 8
#define EBIN_DEFAULT_EPSILON 1e-5f

/* Return codes.  Host-detectable errors are returned synchronously. */
typedef enum ebin_status {
    EBIN_OK = 0,
    EBIN_ERR_INVALID_ARG = 1,         /* NULL handle, NULL buffer with work to do, bad rank/dim */
    EBIN_ERR_UNSUPPORTED_OP = 2,      /* operator code out of range */
    EBIN_ERR_UNSUPPORTED_TYPE = 3,    /* type pair not in the operator's manifest */
    EBIN_ERR_INVALID_ATTR = 4,        /* Mod fmod/opset, BitShift direction */
    EBIN_ERR_INCOMPATIBLE_SHAPES = 5, /* not broadcastable (or not one-way for PRelu/BN/Clip) */
    EBIN_ERR_RANK_TOO_LARGE = 6,      /* an input rank above EBIN_MAX_RANK */
    EBIN_ERR_ALIAS = 7,               /* an input overlaps out without being identical to it */
    EBIN_ERR_CUDA = 8,                /* a CUDA runtime call or kernel launch failed */
    EBIN_ERR_FAMILY = 9               /* a forced loop family cannot traverse this plan */
} ebin_status;

/*
 * Operators.  The nineteen binary operators of "Binary Kernel Design",
 * section "Operators and traversal" (arithmetic, comparisons, logical,
 * bitwise, BitShift, PRelu), plus the two broadcasts that inference
 * BatchNormalization and Clip reduce to (0verkilll/onnx "ops" docs,
 * BatchNormalizationOp and ClipOp; ncnn operators.md, batchnorm and clip).
 * Bias (ncnn operators.md, bias) is EBIN_OP_ADD with B shaped [C,1,1].
 * Then ncnn binaryop's MAX, MIN, RSUB and RDIV, and three fused passes: bias
 * + PReLU, bias + PReLU + BatchNormalization, and the three-input MulAdd.
 */
typedef enum ebin_op {
    EBIN_OP_ADD = 0,
    EBIN_OP_SUB = 1,
    EBIN_OP_MUL = 2,
    EBIN_OP_DIV = 3,
    EBIN_OP_MOD = 4,              /* attrs.fmod; opset 10..28 */
    EBIN_OP_POW = 5,
    EBIN_OP_EQUAL = 6,            /* comparisons write one byte per BOOL (0 or 1) */
    EBIN_OP_LESS = 7,
    EBIN_OP_GREATER = 8,
    EBIN_OP_LESS_OR_EQUAL = 9,
    EBIN_OP_GREATER_OR_EQUAL = 10,
    EBIN_OP_AND = 11,             /* BOOL in, BOOL out; a nonzero byte is true */
    EBIN_OP_OR = 12,
    EBIN_OP_XOR = 13,
    EBIN_OP_BITWISE_AND = 14,
    EBIN_OP_BITWISE_OR = 15,
    EBIN_OP_BITWISE_XOR = 16,
    EBIN_OP_BITSHIFT = 17,        /* attrs.direction */
    EBIN_OP_PRELU = 18,           /* B = slope, broadcast one way to A; a 1-D slope
                                     [C] (C > 1) on A of rank >= 2 is per channel,
                                     axis 1 (0verkilll/onnx ops, PReluOp) */
    EBIN_OP_BATCHNORM = 19,       /* inference; B = [4, C]: scale, bias, mean, var rows,
                                     in A's type or FLOAT32 */
    EBIN_OP_CLIP = 20,            /* B = [2]: {min, max}; attrs.clip_has_min/max */
    /* ncnn operators.md, binaryop operation types 4, 5, 7, 8 (0-3 are ADD..DIV
     * above, 6 = POW is EBIN_OP_POW): */
    EBIN_OP_MAX = 21,             /* IEEE 754-2019 maximum: NaN if either is NaN, +0 > -0 */
    EBIN_OP_MIN = 22,             /* IEEE 754-2019 minimum: NaN if either is NaN, -0 < +0 */
    EBIN_OP_RSUB = 23,            /* B - A */
    EBIN_OP_RDIV = 24,            /* B / A; integer A == 0 raises EBIN_DEVICE_DIV_BY_ZERO */
    /* 0verkilll/onnx ops, ConvPReluOp: the per-output-channel bias add and
     * PReLU of the fused Conv -> PReLU epilogue, as one elementwise pass.
     * B = [2, C]: bias and slope rows, channel axis 1 of A (rank >= 2);
     * y = t >= 0 ? t : slope * t with t = x + bias, binary32 steps rounded
     * once to A's type; floating types only. */
    EBIN_OP_BIAS_PRELU = 25,
    /* 0verkilll/onnx ops, MulAddOp: y = (a * b) + c over three inputs, shapes as
     * the unfused Mul + Add (out = broadcast(broadcast(A, B), C)); binary32
     * product and sum each rounded on their own (no FMA), one rounding to a
     * 16-bit type; integers wrap.  The only three-input operator: plans come
     * from ebin_plan_create3 and run with ebin_execute3. */
    EBIN_OP_MULADD = 26,
    /* The per-channel chain bias add -> PReLU -> inference BatchNormalization
     * as one pass (ConvPReluOp's epilogue followed by BatchNormalizationOp).
     * B = [6, C]: bias, slope, scale, bn_bias, mean, var rows, channel axis 1
     * of A (rank >= 2; rank 2 [N, C] is per element); attrs.epsilon.
     * t = x + bias; t = t >= 0 ? t : slope * t; y = (t - mean) /
     * sqrt(var + eps) * scale + bn_bias: binary32 steps (binary64 for
     * DOUBLE) in the order written, one rounding to A's type; floating types
     * only. */
    EBIN_OP_BIAS_PRELU_BN = 27,
    EBIN_OP_COUNT = 28
} ebin_op;

/* Element types, numbered as ONNX TensorProto.DataType. */
typedef enum ebin_dtype {
    EBIN_FLOAT32 = 1,
    EBIN_UINT8 = 2,
    EBIN_INT8 = 3,
    EBIN_UINT16 = 4,
    EBIN_INT16 = 5,
    EBIN_INT32 = 6,
    EBIN_INT64 = 7,
    EBIN_BOOL = 9,                /* one byte per element */
    EBIN_FLOAT16 = 10,
    EBIN_DOUBLE = 11,             /* computed natively in binary64 */
    EBIN_UINT32 = 12,
    EBIN_UINT64 = 13,
    EBIN_BFLOAT16 = 16
} ebin_dtype;

/*
 * Loop families ("Binary Kernel Design", section "Operators and traversal",
 * loop-family table).  Each has its own kernel; the selection rule is stated
 * at ebin_plan_create.  REPEATED_BLOCK has two: the row kernel when rows are a
 * whole number of 16-byte packs, a flat periodic kernel otherwise.
 */
typedef enum ebin_family {
    EBIN_FAMILY_AUTO = -1,            /* only as a request to ebin_plan_create_forced */
    EBIN_FAMILY_EMPTY = 0,            /* zero output elements: nothing is launched or read */
    EBIN_FAMILY_CONTIGUOUS = 1,
    EBIN_FAMILY_LEFT_SCALAR = 2,
    EBIN_FAMILY_RIGHT_SCALAR = 3,
    EBIN_FAMILY_REPEATED_BLOCK = 4,
    EBIN_FAMILY_INNER_VECTOR_OUTER = 5,
    EBIN_FAMILY_GENERAL_STRIDED = 6
} ebin_family;

/* Device status bits ("Compute, scheduling, and safety": validation before the math). */
#define EBIN_DEVICE_DIV_BY_ZERO 0x1u  /* integer Div/Mod by 0, or integer 0 to a negative power */
#define EBIN_DEVICE_SHIFT_RANGE 0x2u  /* BitShift count >= the element width in bits */

/*
 * Operator attributes.  Pass NULL to ebin_descriptor_create for the defaults
 * (fmod 0, direction LEFT, epsilon 1e-5, both Clip bounds present, no
 * with_scalar).
 *   fmod          Mod only: 0 = floor remainder (result and exact zeros take
 *                 the divisor's sign), 1 = truncated remainder (the dividend's
 *                 sign, including a signed zero).  Floating Mod with fmod 0
 *                 needs opset 28 ("Binary Kernel Design", Operators and
 *                 traversal).
 *   direction     BitShift only: 0 = LEFT, 1 = RIGHT.
 *   epsilon       BatchNormalization and BiasPReluBN only.
 *   clip_has_min  Clip only: nonzero if B[0] is a lower bound.
 *   clip_has_max  Clip only: nonzero if B[1] is an upper bound.
 *   with_scalar   ncnn binaryop's with_scalar (operators.md, binaryop): 1 = B
 *                 is not a tensor but the value scalar_b.  Allowed for Add,
 *                 Sub, Mul, Div, Pow, Max, Min, RSub, RDiv on floating types
 *                 (the page gives b as a float); B is then b rounded to the
 *                 element type (round to nearest even), exactly as a 0-d B
 *                 tensor holding that value.  Plans ignore shape B and read
 *                 no B pointer.  Default 0.
 *   scalar_b      the value b when with_scalar = 1.
 */
typedef struct ebin_attrs {
    int32_t fmod;
    int32_t direction;
    float epsilon;
    int32_t clip_has_min;
    int32_t clip_has_max;
    int32_t with_scalar;
    float scalar_b;
} ebin_attrs;

typedef struct ebin_descriptor_s *ebin_descriptor_t;
typedef struct ebin_plan_s *ebin_plan_t;

/*
 * Build a descriptor ("Binary Kernel Design", Prepared execution: "built once
 * for the node"): checks the operator, opset and attributes, checks that
 * (dtype_a, dtype_b) is a registered type pair of the operator and resolves the
 * output type.  Each descriptor receives a fresh, never reused, monotonic id.
 *
 *   op, opset      operator and the node's opset (only Mod reads opset: 10..28)
 *   attrs          may be NULL (defaults above); copied, not retained
 *   dtype_a/b      element types of A and B; they must be equal, except:
 *                  Pow's exponent B may be any non-BOOL type, and the
 *                  parameter block B of BATCHNORM, BIAS_PRELU and
 *                  BIAS_PRELU_BN may be FLOAT32 beside a FLOAT16, BFLOAT16
 *                  or DOUBLE A (BatchNormalizationOp keeps its parameters in
 *                  a float32 runtime; they enter the chain unrounded,
 *                  widened exactly to DOUBLE for a DOUBLE A).  Such a plan
 *                  keeps the loop family of a same-type block.
 *   out            receives the new descriptor; the caller owns it
 * Errors: INVALID_ARG (out NULL), UNSUPPORTED_OP, UNSUPPORTED_TYPE, INVALID_ATTR.
 */
ebin_status ebin_descriptor_create(ebin_op op, int opset, const ebin_attrs *attrs,
                                   ebin_dtype dtype_a, ebin_dtype dtype_b,
                                   ebin_descriptor_t *out);

/*
 * The descriptor's output element type, resolved when it was built ("Binary
 * Kernel Design", Prepared execution: the descriptor resolves the output type;
 * Compute, scheduling, and safety: comparisons and logical operators write
 * one byte per BOOL): BOOL for the comparisons and And/Or/Xor, else dtype_a.
 * Errors: INVALID_ARG (desc or out NULL).
 */
ebin_status ebin_descriptor_output_dtype(ebin_descriptor_t desc, ebin_dtype *out);

/* The descriptor's monotonic identity (the plan cache keys on it, never on the pointer). */
ebin_status ebin_descriptor_id(ebin_descriptor_t desc, uint64_t *id);

/*
 * Free a descriptor ("Binary Kernel Design", Prepared execution: cache
 * entries are keyed on the descriptor's monotonic id, never its address, so a
 * freed descriptor's plans can never be found again).  Cached plans built
 * from it are dropped from the LRU; plans the caller still holds stay valid
 * (they copy what they need).  NULL is ignored.
 */
void ebin_descriptor_destroy(ebin_descriptor_t desc);

/*
 * Plan the broadcast of concrete input shapes ("Binary Kernel Design",
 * Operators and traversal; Prepared execution for the cache):
 *   1. right-align the shapes (a rank-0 shape is a scalar) and check that each
 *      dimension pair is equal or contains a 1 (0 pairs only with 0 or 1);
 *      PRelu, BatchNormalization, Clip, BiasPRelu and BiasPReluBN broadcast
 *      one way: out == A's shape.  A 1-D PRelu slope [C] with C > 1 on A of
 *      rank >= 2 is per channel (0verkilll/onnx ops, PReluOp): it is read as
 *      [C, 1, ..., 1], which right-aligns onto A's axis 1, so C must equal
 *      shape_a[1];
 *   2. give broadcast dimensions zero strides;
 *   3. drop dimensions of output extent 1;
 *   4. merge adjacent dimensions i, i+1 when stride[i] == stride[i+1] * n[i+1]
 *      holds for A, B and out;
 *   5. pick the loop family:
 *        numel == 0                                   -> EMPTY
 *        rank 1, strides (A,B) (1,1) / (0,1) / (1,0)  -> CONTIGUOUS / LEFT_ / RIGHT_SCALAR
 *        rank 2, one input dense and the other with strides (1,0) (one value
 *        per row) or (0,1) (one row block reused), any row length
 *                                                      -> REPEATED_BLOCK
 *        innermost extent >= 64 and a multiple of the vector width
 *                                                      -> INNER_VECTOR_OUTER
 *        otherwise                                     -> GENERAL_STRIDED
 *      (vector width = 16 bytes / element size of A).
 * The result is looked up in, or inserted into, a process-wide LRU of
 * EBIN_PLAN_CACHE_CAPACITY plans keyed on (descriptor id, types, both shapes);
 * a miss always builds and validates a fresh plan.
 *
 * Shapes: shape_a[rank_a], shape_b[rank_b], dims >= 0.  For BatchNormalization
 * B is [4, C], for BiasPRelu [2, C] and for BiasPReluBN [6, C], with
 * C == shape_a[1] (rank_a >= 2); for Clip B is [2].  Each input's element
 * count and the output's stay below 2^60 (EBIN_MAX_ELEMENTS), so that every
 * element offset and byte size fits in int64_t; a shape with a zero extent is
 * empty whatever its other extents.
 *   out            receives a plan reference; release it with ebin_plan_release
 * Errors: INVALID_ARG (also an element count of 2^60 or more),
 * RANK_TOO_LARGE, INCOMPATIBLE_SHAPES.
 */
ebin_status ebin_plan_create(ebin_descriptor_t desc, const int64_t *shape_a, int rank_a,
                             const int64_t *shape_b, int rank_b, ebin_plan_t *out);

/*
 * As ebin_plan_create, but force a loop family (for testing every kernel on
 * the same inputs).  Forced plans bypass the cache.  GENERAL_STRIDED can run
 * every plan; the others only geometries they can traverse (else FAMILY).
 * A with_scalar plan runs only its own family or GENERAL_STRIDED.  With zero
 * output elements the family is always EMPTY.
 */
ebin_status ebin_plan_create_forced(ebin_descriptor_t desc, const int64_t *shape_a, int rank_a,
                                    const int64_t *shape_b, int rank_b, ebin_family family,
                                    ebin_plan_t *out);

/*
 * Plan for strided input views: inputs need not be dense.
 * strides_a / strides_b give each input's element strides in its own rank
 * (non-negative; NULL = dense row-major); strides equal to the dense ones are
 * the dense plan.  The planner uses the view's strides in place of the dense
 * ones, then drops unit dims and merges dims exactly as for dense inputs.  The
 * vector families additionally need every row of a packed input to start on a
 * 16-byte boundary (its outer strides multiples of 16 bytes of elements), else
 * the plan is GENERAL_STRIDED.  B strides are refused (INVALID_ARG) for the
 * parameter blocks of BatchNormalization, Clip, BiasPRelu and BiasPReluBN, and ignored with
 * with_scalar.  family: EBIN_FAMILY_AUTO (the plan is cached, keyed with the
 * strides) or a forced family as ebin_plan_create_forced (not cached).
 * A view's storage extent (largest offset + 1) stays below 2^60, as element
 * counts do (else INVALID_ARG).
 * A strided input is never executed in place: any overlap with out is ALIAS.
 * ebin_execute_host copies each input's whole storage extent (largest offset
 * + 1 elements) and runs strided plans without the chunked pipeline.
 * Errors: as ebin_plan_create, and FAMILY for a forced family.
 */
ebin_status ebin_plan_create_strided(ebin_descriptor_t desc, const int64_t *shape_a,
                                     const int64_t *strides_a, int rank_a,
                                     const int64_t *shape_b, const int64_t *strides_b, int rank_b,
                                     ebin_family family, ebin_plan_t *out);

/*
 * Plan a three-input operator (MulAdd): the three shapes broadcast together
 * (NumPy rules, right-aligned; the output is broadcast(broadcast(A, B), C)),
 * unit dims are dropped and adjacent dims merged where all three stride sets
 * allow.  Loop family: a row traversal (reported as CONTIGUOUS at rank 1 with
 * three dense inputs, RIGHT_SCALAR at rank 1 otherwise, INNER_VECTOR_OUTER at
 * rank >= 2) when every input moves along the innermost dim with stride 0 or
 * 1, that dim is a multiple of 16 bytes of elements and, at rank >= 2, at
 * least 64 long; else GENERAL_STRIDED.  Plans are cached like two-input plans,
 * keyed on all three shapes.  The _forced form accepts AUTO, GENERAL_STRIDED or
 * the family the plan would pick, and bypasses the cache.
 * Errors: INVALID_ARG (also for a two-input descriptor), RANK_TOO_LARGE,
 * INCOMPATIBLE_SHAPES, FAMILY.  ebin_plan_create refuses three-input
 * descriptors with INVALID_ARG.
 */
ebin_status ebin_plan_create3(ebin_descriptor_t desc, const int64_t *shape_a, int rank_a,
                              const int64_t *shape_b, int rank_b, const int64_t *shape_c,
                              int rank_c, ebin_plan_t *out);
ebin_status ebin_plan_create3_forced(ebin_descriptor_t desc, const int64_t *shape_a, int rank_a,
                                     const int64_t *shape_b, int rank_b, const int64_t *shape_c,
                                     int rank_c, ebin_family family, ebin_plan_t *out);

/*
 * The plan's output shape ("Binary Kernel Design", Operators and traversal:
 * the right-aligned broadcast takes, per dimension, the extent that is not 1;
 * one-way operators keep A's shape).  `shape` must hold EBIN_MAX_RANK entries;
 * *rank receives its rank (0 for a scalar).  Errors: INVALID_ARG (a NULL
 * argument).
 */
ebin_status ebin_plan_output_shape(ebin_plan_t plan, int64_t *shape, int *rank);

/* Number of output elements. */
ebin_status ebin_plan_numel(ebin_plan_t plan, int64_t *numel);

/*
 * The loop family the plan selected ("Binary Kernel Design", Operators and
 * traversal, loop-family table; the rule is stated at ebin_plan_create).
 * Execution may still run a 16-byte-vector family's plan on the general
 * kernel when a buffer is off 16-byte alignment.  Errors: INVALID_ARG.
 */
ebin_status ebin_plan_family(ebin_plan_t plan, ebin_family *family);

/*
 * The coalesced traversal: *rank dims with extents n[] and element strides of
 * A and B (0 on broadcast dims); out is dense.  Arrays hold EBIN_MAX_RANK.
 * A plan without output elements reports rank 1, n[0] = 0 and zero strides.
 */
ebin_status ebin_plan_geometry(ebin_plan_t plan, int *rank, int64_t *n, int64_t *stride_a,
                               int64_t *stride_b);

/*
 * Drop one reference ("Binary Kernel Design", Prepared execution: plans live
 * in a bounded LRU and are rebuilt on a miss; a plan evicted while a caller
 * holds it stays valid for that caller).  The plan is freed when no caller and
 * no cache slot holds it.  NULL is ignored.
 */
void ebin_plan_release(ebin_plan_t plan);

/* Plan cache counters since the last clear, and its current size (<= 8). */
ebin_status ebin_plan_cache_stats(uint64_t *hits, uint64_t *misses, int *size);

/* Empty the plan cache and zero its counters (held plans stay valid). */
void ebin_plan_cache_clear(void);

/*
 * Run a plan on device buffers ("Binary Kernel Design", Compute, scheduling,
 * and safety): one kernel of the plan's family is enqueued on `stream`.
 *   A, B, out   device pointers of the plan's input and output shapes (dense).
 *               B may be NULL only for Clip without bounds.  With zero output
 *               elements nothing is read or written and NULL is accepted.
 *               An input may alias out only if it is the same pointer and has
 *               the output's type and shape; any other overlap is ALIAS.
 *               Pointers not aligned to 16 bytes run the general kernel.
 *   stream      cudaStream_t as void* (NULL = legacy default stream)
 * Returns once the kernel is enqueued.  Invalid elements (integer division by
 * zero, shift counts out of range) do not stop the kernel: they write 0 and set
 * bits in the stream's status word, read with ebin_get_device_status.  That
 * word (4 bytes of device memory per stream handle and device) is allocated by
 * the first validating operator on the stream and kept until the process
 * exits; a later stream that reuses the handle's value reuses the word.
 * Stream capture: the launch path makes no allocation and no synchronising
 * call, so executions can be captured into a CUDA graph and replayed.  The one
 * exception is the first validating operator on a stream, which allocates that
 * stream's status word: run one on the capturing stream before the capture
 * begins.  Launch the kernels once before the first capture, because a
 * kernel's first launch loads its module (and, for the per-row kernels, looks
 * up its occupancy once to size the grid).
 * Errors: INVALID_ARG, ALIAS, CUDA.
 */
ebin_status ebin_execute(ebin_plan_t plan, const void *A, const void *B, void *out,
                         void *stream);

/*
 * Run a three-input plan: out = op(A, B, C) on device buffers, enqueued on
 * `stream`.  A, B, C are dense in their own shapes; each may be `out` only as
 * the identical buffer with the output's element count (anything else
 * overlapping out is ALIAS).  Pointers off 16-byte alignment run the general
 * kernel.  A two-input plan, or NULL buffers with work to do, give INVALID_ARG.
 * Errors: INVALID_ARG, ALIAS, CUDA.
 */
ebin_status ebin_execute3(ebin_plan_t plan, const void *A, const void *B, const void *C,
                          void *out, void *stream);

/*
 * End-to-end form of ebin_execute for callers whose data lives in host
 * memory: copies host_a -> dev_a and host_b -> dev_b, runs the kernel, and
 * copies dev_out -> host_out.  All six buffers belong to the caller and are
 * sized for the plan (host_b / dev_b NULL where ebin_execute takes B = NULL);
 * host buffers should be pinned for the copies to run asynchronously.
 *
 * Contiguous and scalar-family plans of at least 2^21 elements run as a
 * pipeline: the output range is cut into at most 32 chunks (multiples of 4096
 * elements, at least 2^20), and chunk c+1 is copied in while chunk c computes
 * on `stream` and chunk c-1 is copied out.  The copies go on two streams per
 * device that the library creates on first use and keeps; events order them
 * after the work already queued on `stream`, and `stream` itself waits for the
 * last output copy.  Other plans enqueue copies, kernel and copy-back on
 * `stream` one after another.
 *
 * Does not synchronise: host_out is valid once `stream` has completed.
 * Errors as ebin_execute (checks on the device buffers), and INVALID_ARG for
 * host_b without dev_b.
 */
ebin_status ebin_execute_host(ebin_plan_t plan, const void *host_a, const void *host_b,
                              void *host_out, void *dev_a, void *dev_b, void *dev_out,
                              void *stream);

/*
 * End-to-end form without staging: the kernel reads host_a and host_b and
 * writes host_out in place, over the host-device link.  On Grace-Blackwell
 * this link is NVLink-C2C, and the kernel keeps it busy in both directions
 * at once.  Same computation and results as ebin_execute.  No counterpart in
 * the pages: they only speak of device buffers.
 *
 * Each host buffer must lie wholly inside one pinned allocation mapped into
 * the device's address space: cudaHostAlloc / cudaMallocHost memory, or
 * memory registered with cudaHostRegister, which on a unified-addressing
 * system is mapped.  For each buffer, the first and last byte of its extent
 * are checked: both must be host memory, carry the same allocation id and
 * map contiguously.  A buffer that fails the check (pageable memory, a range
 * past its allocation) gives INVALID_ARG before any device work, so the
 * kernel never touches an unmapped address.  The extents are: A and B their
 * storage extent in elements of their types; out the output's element count
 * in the output type.  host_b is NULL where ebin_execute takes B = NULL.
 *
 * Enqueued on `stream`; does not synchronise.  host_out is valid once
 * `stream` has completed, and the host must not touch the buffers before
 * then.
 * Errors: as ebin_execute, and INVALID_ARG for an unmapped buffer.
 */
ebin_status ebin_execute_mapped(ebin_plan_t plan, const void *host_a, const void *host_b,
                                void *host_out, void *stream);

/*
 * ebin_execute3 on host buffers, in place over the host-device link, with the
 * checks of ebin_execute_mapped on all four buffers (each input's extent is
 * its element count in the plan's type).  A two-input plan gives INVALID_ARG.
 * Errors: as ebin_execute3, and INVALID_ARG for an unmapped buffer.
 */
ebin_status ebin_execute3_mapped(ebin_plan_t plan, const void *host_a, const void *host_b,
                                 const void *host_c, void *host_out, void *stream);

/*
 * Read and clear the device status word of `stream` on the current device
 * ("Binary Kernel Design", Compute, scheduling, and safety: invalid inputs --
 * integer division or modulo by zero, shift counts -- are found by validation
 * before the math; here each kernel records them as bits instead of
 * stopping): synchronises the stream, returns the OR of the EBIN_DEVICE_*
 * bits raised since the last call, then zeroes the word (stream-ordered).  A
 * stream that never ran a validating operator reports 0.
 * Errors: INVALID_ARG (bits NULL), CUDA.
 */
ebin_status ebin_get_device_status(void *stream, uint32_t *bits);

/*
 * Execute without any allocation by the library.  No counterpart in the pages:
 * this entry point exists for callers that cannot let a library allocate
 * device memory -- an application whose device memory is wholly owned by its
 * own arena allocator, a plugin whose host framework forbids allocation while
 * work is being enqueued, or a latency-critical loop that cannot absorb the
 * implicit synchronisation of cudaMalloc.  ebin_execute would cudaMalloc a
 * per-stream status word the first time a validating operator (integer Div,
 * Mod, Pow; BitShift) runs on a stream; this call runs the same kernels with
 * the status word taken from a fixed array compiled into the library instead
 * (EBIN_NOALLOC_STATUS_SLOTS words = 256 bytes, held on every device that
 * loads the library until the process exits).
 *
 *   plan, A, B, out, stream   as for ebin_execute (same checks and errors)
 *   status_slot               which word of the array this call uses,
 *                             0 <= slot < EBIN_NOALLOC_STATUS_SLOTS; anything
 *                             else returns EBIN_ERR_INVALID_ARG
 *   status_bits               NULL, or a host word that receives the
 *                             EBIN_DEVICE_* bits of this call; with a non-NULL
 *                             pointer the call waits for `stream` to finish.
 *                             With NULL the bits stay in the slot, to be read
 *                             later with ebin_noalloc_read_status.
 * The checks, the kernel choice and the alignment fallback are ebin_execute's
 * own (one shared implementation).  The slot is zeroed (stream-ordered) at the
 * start of every call, so it holds the bits of the last call that used it.
 * All calls share the array: calls that use the same slot and overlap on the
 * GPU race on it.  The first call on a device looks up the array's device
 * address once (cudaGetSymbolAddress), so make that first call before any
 * stream capture.  Nothing here calls cudaMalloc, cudaFree or any allocating
 * routine.
 */
#define EBIN_NOALLOC_STATUS_SLOTS 64
ebin_status ebin_execute_noalloc(ebin_plan_t plan, const void *A, const void *B, void *out,
                                 void *stream, int status_slot, uint32_t *status_bits);

/*
 * Read one word of ebin_execute_noalloc's status array on the current device,
 * without allocating.  No counterpart in the pages.  Waits for the work
 * already queued on `stream` (the stream the calls that used the slot ran on,
 * or one ordered after them), then returns in *bits the EBIN_DEVICE_* bits of
 * the last ebin_execute_noalloc call that used `status_slot`; the slot is not
 * cleared (the next call that uses it clears it).  A slot no call has used
 * reads 0.  Like ebin_execute_noalloc, the first use on a device looks up the
 * array's address.
 * Errors: INVALID_ARG (bits NULL, or a slot outside [0, EBIN_NOALLOC_STATUS_SLOTS)),
 * CUDA.
 */
ebin_status ebin_noalloc_read_status(int status_slot, void *stream, uint32_t *bits);

/* Kernels this library has launched in this process (for launch accounting). */
uint64_t ebin_launch_count(void);

/* Bytes per element of a type (0 if unknown). */
size_t ebin_dtype_size(ebin_dtype dtype);

/*
 * A static, human-readable name for a status code ("Binary Kernel Design",
 * Compute, scheduling, and safety: invalid inputs are reported, not acted
 * on).  Unknown codes give "unknown status".  Never NULL; not to be freed.
 */
const char *ebin_status_string(ebin_status status);

#ifdef __cplusplus
}
#endif

#endif /* EBIN_H */
