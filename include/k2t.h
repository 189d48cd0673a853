/*
 * k2t.h -- C ABI of the k^2-tree semiring SpMV library (GB300, sm_103a).
 *
 * The operations follow "A GPU Engine for Sparse Matrix-Vector Products on
 * k^2-Tree-Compressed Graphs" (Tosoni & Mencagli):
 *   - the k^2-tree of a Boolean n x n matrix, n = 2^l, stored pointer-free
 *     level by level as signatures of k^2 bits, bit b of a node set iff its
 *     quadrant b = 2*b1 + b0 is non-empty (section 2.1, Figure 1);
 *   - y = A x and y^T = x^T A over a semiring (section 2.2, Table 1;
 *     section 3.6), for one vector or a batch of B vectors (section 3.6);
 *   - the level-synchronous traversal of Algorithm 1 (section 3), child
 *     offsets from a scan or a sampled directory (section 3.2), a host-side
 *     top, tiles (section 3.4), tree-only and cached-frontier configurations
 *     (section 3.5);
 *   - the device memory of a product fixed before any kernel runs
 *     (section 1, "Our approach"; section 3.4).
 *
 * Conventions shared by every call
 *   - Every function returns K2T_OK (0) or a negative K2T_E* status; none
 *     aborts the process.  k2t_strerror() names a status.
 *   - A k2t_tree is opaque and owned by the library; k2t_free() releases its
 *     host memory and any device memory the library allocated for it.
 *   - Device pointers (x, y, the arena) belong to the caller, who keeps them
 *     alive until the work queued on the given stream has finished.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Device calls are asynchronous on that stream.
 *   - Vector layout: row-major n x B fp32 (B contiguous values per vertex),
 *     or, for the Boolean semiring, one uint32 word per vertex whose bit b
 *     is vector b (B <= 32).  Right products read n_cols entries and write
 *     n_rows; left products the reverse.  x and y must not overlap.
 *   - Host calls are thread-compatible: one thread at a time per tree.
 *   - Products of one tree must not overlap on the GPU: the tree's arena
 *     holds per-product scratch (level-synchronous frontier buffers, the
 *     sums of heavy plus-times outputs).  Queue them on one stream, or order
 *     the streams.  Different trees are independent.
 */
#ifndef K2T_H
#define K2T_H

#include <stdint.h>

/* Only the calls below are exported: the library is built with hidden
 * symbol visibility, so its C++ internals (template instances and their
 * function-local state) stay private to each library file, and two builds
 * (libk2t.so and the bounds-checked libk2t_checked.so) can be loaded into one
 * process side by side. */
#if defined(__GNUC__)
#define K2T_API __attribute__((visibility("default")))
#else
#define K2T_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define K2T_OK        0
#define K2T_EINVAL   (-1)  /* bad argument: null pointer, bad enum, misaligned vector */
#define K2T_ERANGE   (-2)  /* id >= n, side > 2^32, batch > limit, level too wide */
#define K2T_ENOMEM   (-3)  /* host or device allocation failed, or arena too small */
#define K2T_ECUDA    (-4)  /* a CUDA runtime call failed (see k2t_last_cuda_error) */
#define K2T_ESTATE   (-5)  /* wrong call order, e.g. a product before k2t_upload */
#define K2T_EDEVICE  (-6)  /* a device-side consistency check failed */
#define K2T_ETIMEOUT (-7)  /* a device-side wait ran out of iterations */

/* Device status word.  The first 4 bytes of a tree's arena (k2t_upload)
 * hold a word that kernels set instead of trapping: bit 0 when a bounded
 * wait for a staged copy ran out (the block that waited left its outputs
 * untouched), bit 1 when a checked build found an index out of range.
 * Synchronising calls (k2t_spmv_host, k2t_msbfs) read it after their work
 * and return K2T_ETIMEOUT (bit 0) or K2T_EDEVICE (other bits); the word is
 * sticky until k2t_status() clears it.  Asynchronous calls leave the check
 * to the caller (k2t_status after the stream's work). */
#define K2T_STATUS_WAIT_TIMEOUT 1u
#define K2T_STATUS_OUT_OF_RANGE 2u

/* Opaque handle to one built tree (host image, plan and device image). */
typedef struct k2t_tree k2t_tree;

/* ---- enums ------------------------------------------------------------- */
#define K2T_RIGHT 0          /* y = A x        (section 2.2)                 */
#define K2T_LEFT  1          /* y^T = x^T A    (section 3.6)                 */

#define K2T_PLUS_TIMES 0     /* (R, +, x, 0, 1): contribution w * x_j        */
#define K2T_BOOLEAN    1     /* ({0,1}, or, and): contribution x_j's word    */
#define K2T_MIN_PLUS   2     /* (R u {inf}, min, +, inf, 0): w + x_j          */

/* Engines: how a product walks the tree. */
#define K2T_ENGINE_AUTO      0  /* CACHED if the last level is cached, else FUSED      */
#define K2T_ENGINE_FUSED     1  /* tree-only, one launch: each warp descends a chunk
                                   of whole subtrees (at most chunk_cap leaves) in
                                   shared memory                                      */
#define K2T_ENGINE_LEVELSYNC 2  /* tree-only, Algorithm 1 as written: one expand
                                   launch per tile and level into global frontier
                                   buffers of at most tile_M codes (section 3.4)      */
#define K2T_ENGINE_CACHED    3  /* k^2+F: one leaf kernel over the cached
                                   coordinates of the last internal level (3.5)       */
#define K2T_ENGINE_BANDED    4  /* k^2+F ordered by row band: the cached level is
                                   kept grouped by bands of band_rows rows, so a
                                   thread block owns a band and keeps its part of
                                   y (right product) or x (left product) in
                                   shared memory: one scattered access per edge
                                   instead of two                                    */

/* ChildOffset source (section 3.2), used by the LEVELSYNC engine. */
#define K2T_OFFSETS_DIRECTORY 0 /* one sample per 256 nodes, stored with the tree  */
#define K2T_OFFSETS_SCAN      1 /* prefix sums of fan-outs computed at each product */

#define K2T_MAX_LEVELS 33
#define K2T_MAX_BATCH  32

/* ---- options ----------------------------------------------------------- */
typedef struct {
    uint32_t n_k4_levels;         /* leading levels with k = 4 (hybrid tree); 0 = k = 2 throughout */
    uint32_t cache_last_internal; /* 1: keep the coordinates of the last internal level (k^2+F)    */
    uint32_t engine;              /* K2T_ENGINE_*                                                   */
    uint32_t offsets;             /* K2T_OFFSETS_* (LEVELSYNC only; the other engines use the
                                     directory or the chunk plan)                                   */
    uint32_t host_top_max_nodes;  /* products start at the deepest level with at most this many
                                     nodes, expanded on the host (section 3.4); default 65536       */
    uint32_t chunk_cap;           /* FUSED: leaves per chunk, the part of the tree one warp
                                     descends (a chunk's widest level); default 256, from 4 to 512  */
    uint64_t tile_m;              /* LEVELSYNC: children per tile M; default 2^20, at least 4      */
    uint32_t max_batch;           /* largest B products will use (1..32); sizes host-vector buffers */
    uint32_t host_vectors;        /* 1: the workspace also holds device x and y of max_batch
                                     vectors for k2t_spmv_host                                      */
    uint32_t use_graph;           /* LEVELSYNC: record a product's launches once as a CUDA graph   */
    uint32_t threads;             /* host threads for k2t_build; 0 = all cores                     */
    uint32_t band_rows;           /* BANDED: rows per band (power of two, 16..65536); default 4096 */
    uint32_t band_cols;           /* BANDED: columns per tile (power of two >= 16); default 2^23;
                                     0 = one column band                                             */
    uint32_t heavy_terms;         /* plus-times: the most non-zeros one fp32 sum may hold.  An
                                     output with more non-zeros in its row (right) or column
                                     (left), counted over the input list, is "heavy": summed as
                                     heavy_mode says and rounded to fp32 once.  Default 160 (0 =
                                     default), the largest count for which an fp32 sum meets the
                                     plus-times bound in any order; 0xffffffff = never (every
                                     output one fp32 sum).  See "Accumulation precision" below.   */
    uint32_t heavy_mode;          /* how heavy outputs are summed: 0 (default) in fp32 partial
                                     sums of at most heavy_terms terms each (the builder picks
                                     2^bits of them per output and checks the count of every
                                     one), added in fp64 at the end; 1 in fp64 (fp64 atomics;
                                     slower).  See "Accumulation precision" below.                */
    uint32_t leaf_k;              /* side of a leaf block: 0 (default: chosen by the build), 2 or
                                     4.  4: the leaf level stores 4x4 bitmaps (16-bit signatures,
                                     cell (dr, dc) at bit 4*dr + dc), the larger leaves of section
                                     5.6; every other level keeps k = 2 (or k = 4 on the n_k4 top
                                     levels).  0 picks 4 when 2x2 leaves would hold at least 1.75
                                     non-zeros each on average, else 2.  4x4 leaves need the
                                     FUSED or CACHED engine (AUTO resolves to one of them);
                                     LEVELSYNC and BANDED give EINVAL for 4 and use 2 for 0.      */
    uint32_t reserved[3];
} k2t_opts;

/* ---- statistics -------------------------------------------------------- */
typedef struct {
    uint64_t n_rows, n_cols;      /* matrix shape as given                        */
    uint64_t nnz;                 /* distinct non-zeros (= set bits of L)          */
    uint32_t levels;              /* l: levels 0 (root) .. l-1 (leaves)            */
    uint32_t n_k4_levels;
    uint32_t dim_bits;            /* padded side n = 2^dim_bits                    */
    uint32_t d0;                  /* first level a product expands on the device   */
    uint64_t level_nodes[K2T_MAX_LEVELS];
    uint64_t tree_bits;           /* |T| + |L| over all levels                     */
    uint64_t t_bytes_device;      /* signature bytes of levels d0..l-2 on device   */
    uint64_t l_bytes_device;      /* leaf signature bytes on device                */
    uint64_t dir_bytes;           /* directory samples on device                   */
    uint64_t top_bytes;           /* coordinates of level d0 on device             */
    uint64_t cached_bytes;        /* cached coordinates of level l-2 (k^2+F; banded:
                                     coordinates, first-leaf offsets, signatures)  */
    uint64_t plan_bytes;          /* chunk table / root coordinates (FUSED)        */
    uint64_t scratch_bytes;       /* frontier buffers and scan space (LEVELSYNC)   */
    uint64_t vector_bytes;        /* device x and y for k2t_spmv_host              */
    uint64_t workspace_bytes;     /* total = k2t_workspace_bytes                   */
    uint64_t n_chunks;            /* FUSED chunks                                  */
    uint64_t n_steps;             /* LEVELSYNC launches per product (tiles x kinds)*/
    uint32_t engine;              /* resolved engine                               */
    uint32_t offsets;
    uint32_t uploaded;            /* 1 after k2t_upload                            */
    uint32_t heavy_rows;          /* heavy outputs of right products               */
    uint32_t heavy_cols;          /* heavy outputs of left products                */
    uint32_t heavy_kib;           /* device KiB of the heavy outputs' tables and
                                     sums (part of workspace_bytes)                */
    uint32_t leaf_k;              /* side of a leaf block: 2 or 4                  */
    uint32_t heavy_fp64[2];       /* heavy outputs summed in fp64 (right, left)    */
    uint32_t heavy_max_terms[2];  /* most terms one fp32 partial sum of a heavy
                                     output receives (right, left)                 */
    uint32_t pad;
    uint64_t heavy_partials[2];   /* fp32 partial sums of the heavy outputs
                                     (right, left)                                 */
} k2t_stats;

/* Fill *o with the defaults: k = 2, tree-only FUSED engine (AUTO), directory
 * offsets, top of at most 2^16 nodes, chunk_cap 256, tile_m 2^20,
 * max_batch 32, no host vectors, CUDA graph on, all host threads, leaf size
 * chosen by the build, heavy_terms 160 in fp32 partial sums. */
K2T_API void k2t_default_opts(k2t_opts *o);

/* Build the tree of the n_rows x n_cols Boolean matrix whose non-zeros are
 * (rows[i], cols[i]), i < nnz, on the host (section 2.1; construction is the
 * host step of section 5.1).  Duplicated pairs count once.  The side is padded
 * to 2^b (at least 4, at least 2^(2*n_k4+2), with 4x4 leaves 2^(2*n_k4+3)),
 * giving b - n_k4 levels (4x4 leaves: b - n_k4 - 1).  The COO arrays are read, not
 * kept.  opts may be NULL (defaults).  Plans the product as well: host-side
 * top (3.4), directories (3.2), chunk or tile plan (3.4), cached level (3.5).
 * Errors: EINVAL (null out/arrays with nnz > 0, zero side, bad option),
 * ERANGE (an id >= its side, side > 2^32, a level wider than 2^32 - 1 nodes),
 * ENOMEM.  On error *out is NULL. */
K2T_API int k2t_build(const uint32_t *rows, const uint32_t *cols, uint64_t nnz,
              uint64_t n_rows, uint64_t n_cols, const k2t_opts *opts, k2t_tree **out);

/* Exact device bytes k2t_upload places in its arena (tree, directory, top,
 * cached level, plan, scratch, the heavy outputs' tables and sums,
 * optional host-product vectors), known before
 * any kernel runs (section 1, "Our approach").  Dense x and y of device
 * products are the caller's and not included. */
K2T_API int k2t_workspace_bytes(const k2t_tree *t, uint64_t *bytes);

/* Copy the device image into `arena` (device memory of at least
 * k2t_workspace_bytes, 256-byte aligned) or, if arena is NULL, into one
 * cudaMalloc of exactly that size that the library owns.  Uploading twice
 * is ESTATE.  Errors: EINVAL (misaligned arena), ENOMEM (arena_bytes too
 * small or allocation failure), ECUDA. */
K2T_API int k2t_upload(k2t_tree *t, void *arena, uint64_t arena_bytes, void *stream);

/* y = A x (dir K2T_RIGHT) or y^T = x^T A (K2T_LEFT) over `semiring` with edge
 * weight w (Table 1: plus-times w = 1, tropical w = 1 for hop counts; the
 * Boolean semiring ignores w), for B vectors, on device buffers, queued on
 * `stream`.  y is overwritten with the semiring zero first (Algorithm 1,
 * line 1).  Boolean and tropical results are exact and deterministic.
 * Tropical minima follow the IEEE total order without NaN (-0 < +0); NaN
 * inputs give unspecified values.
 * Accumulation precision (plus-times): sums run in no fixed order, and
 * every output meets |y - y_ref| <= 1e-5 * sum_j |w x_j| + 1e-6 (y_ref the
 * exact sum) for any finite inputs whose partial sums stay in the fp32
 * range.  An fp32 sum of N terms w*x_j (each rounded once), formed by any
 * tree of additions, errs by at most N * 2^-24 * sum|w x_j| (to first
 * order), which is within 1e-5 for N <= 167.  So an output with at most
 * opts.heavy_terms (default 160) non-zeros is one fp32 sum, reduced in warp
 * windows or in y; a heavy output (more non-zeros) is summed in fp32 partial
 * sums of at most heavy_terms terms each (heavy_mode 0) or in fp64 (mode 1),
 * then the partial sums are added in fp64 and rounded to fp32 once, at the
 * end of the product: at most (heavy_terms + 1) * 2^-24 of the sum.
 * Heavy outputs need B <= opts.max_batch.
 * x and y must be 4-byte aligned (16-byte alignment enables vector access).
 * The tree's device (current at k2t_upload) must be the current device.
 * Errors: ESTATE (not uploaded, or another device current), EINVAL (bad
 * dir/semiring, null, B = 0, overlap), ERANGE (B > 32; plus-times with heavy
 * outputs and B > opts.max_batch), ECUDA (launch failure). */
K2T_API int k2t_spmv(k2t_tree *t, int32_t dir, int32_t semiring, float w,
             const void *x, void *y, uint32_t B, void *stream);

/* k2t_spmv that also records the cudaEvent_t `event_after_fill` on the stream
 * between the fill of y and the product kernels, so a caller can time the
 * two apart with CUDA events.  When the level-synchronous engine replays a
 * CUDA graph the event is recorded before the graph (it then marks the start
 * of the whole product).  Same errors as k2t_spmv. */
K2T_API int k2t_spmv_marked(k2t_tree *t, int32_t dir, int32_t semiring, float w,
                    const void *x, void *y, uint32_t B, void *stream, void *event_after_fill);

/* Same product on HOST buffers: copies x to the device vectors of the
 * workspace, runs k2t_spmv, copies y back, and synchronises the stream.
 * Needs opts.host_vectors = 1 and B <= opts.max_batch (else ESTATE/ERANGE).
 * Host buffers may be pageable; pinned buffers copy faster.  After the copy
 * back it reads the device status word: ETIMEOUT or EDEVICE if it is set. */
K2T_API int k2t_spmv_host(k2t_tree *t, int32_t dir, int32_t semiring, float w,
                  const void *x_host, void *y_host, uint32_t B, void *stream);

/* The level-synchronous product of k2t_spmv for callers that cannot call
 * cudaMalloc: a framework that owns all device memory through its own pool,
 * code that must never synchronise the device, or code held to a memory
 * budget fixed before it starts.  The pages have no counterpart; it is an
 * addition of this library.  It allocates nothing: its frontier buffers and
 * scan space live in one file-scope device array of
 * k2t_noalloc_scratch_limit() bytes (64 MiB), which every GPU that loads the
 * library holds until the process exits.  The caller provides the uploaded
 * tree (its arena may come from k2t_upload with a caller-owned buffer), x and
 * y, with the layout and results of k2t_spmv.
 *   - The tree must use the LEVELSYNC engine (else ESTATE) and its frontier
 *     buffers plus scan space must fit the array (else ERANGE; lower
 *     opts.tile_m to fit).
 *   - The tree's device (current at k2t_upload) must be current (else
 *     ESTATE).
 *   - The first call on a device, with that device current, looks up the
 *     array's device address (cudaGetSymbolAddress); make that first call
 *     before any stream capture.
 *   - Every call shares the array.  Nothing in it needs to start at zero;
 *     calls whose work overlaps on the GPU race on it, so order them (one
 *     stream, or events).
 *   - k2t_workspace_bytes still counts the level-synchronous scratch in the
 *     tree's arena, which this call leaves unused: the device memory in use
 *     is the workspace plus the 64 MiB array.
 *   - Other errors as k2t_spmv. */
K2T_API int k2t_spmv_noalloc(k2t_tree *t, int32_t dir, int32_t semiring, float w,
                     const void *x, void *y, uint32_t B, void *stream);

/* Read the tree's device status word (see "Device status word"): waits for
 * the work queued on `stream`, stores the word in *word and, if clear != 0,
 * resets it to 0.  Returns K2T_OK, or ESTATE (not uploaded), EINVAL (null),
 * ECUDA. */
K2T_API int k2t_status(k2t_tree *t, uint32_t *word, int32_t clear, void *stream);

/* Size in bytes of the device array k2t_spmv_noalloc works in. */
K2T_API uint64_t k2t_noalloc_scratch_limit(void);

/* Boolean product C = A B of two trees: A n x m, B m x p (a->n_cols ==
 * b->n_rows), built with the same padded side and k = 2 on every level
 * (n_k4_levels = 0, leaf_k = 2).  Section 7 of the pages: a level-synchronous
 * descent over a frontier of node pairs (node of A, node of B, same level,
 * matching inner block) expanding into the matching quadrant sub-products;
 * at the leaves, 2x2 Boolean products.  Runs on the current device on
 * `stream` (the trees need not be uploaded; the product copies every level's
 * signatures and directory to memory it allocates and frees), then builds C
 * on the host with k2t_build(opts) into *out (caller frees with k2t_free).
 * Errors: EINVAL (null, shapes or tree kinds that do not match), ENOMEM,
 * ECUDA, and k2t_build's errors. */
K2T_API int k2t_bool_product(const k2t_tree *a, const k2t_tree *b, const k2t_opts *opts, k2t_tree **out, void *stream);

/* Transitive closure A+ (pairs joined by a path of one or more edges) of a
 * square tree by repeated squaring, C <- C or C C (section 7), until C stops
 * growing or max_iters squarings ran; *iters = squarings run.  *out is C's
 * tree built with opts (an automatic leaf size resolves to 2x2 leaves, which
 * every squaring needs).  Errors as k2t_bool_product; EINVAL for a
 * non-square tree. */
K2T_API int k2t_bool_closure(const k2t_tree *a, const k2t_opts *opts, uint32_t max_iters, k2t_tree **out,
                     uint32_t *iters, void *stream);

/* Multi-source breadth-first search to the fixed point (section 5.8): hop
 * distances from B <= 32 sources at once, one batched Boolean product per
 * level, with a mark kernel over dense n x B tables.  dir K2T_RIGHT: vertex i
 * is reached from j when A_ij = 1 (the product y = A x over the frontier);
 * K2T_LEFT: vertex j is reached from i when A_ij = 1 (y^T = x^T A).  The
 * matrix must be square.
 *   sources   host array of B vertex ids (< n)
 *   dist      device int32 array, n x B row-major: the level at which vertex v
 *             is first reached from source b, or -1 if never (within
 *             max_levels); dist[s_b][b] = 0
 *   work      device buffer of k2t_msbfs_work_bytes(t) bytes (frontier,
 *             visited, product output, counter), owned by the caller
 *   levels    out: levels run (the last one reached no new vertex, or the cap)
 * Synchronises the stream once per level (to read the new-vertex count and
 * the device status word).
 * Errors: ESTATE (not uploaded), EINVAL (non-square, bad dir, null),
 * ERANGE (B = 0 or > 32, a source >= n), ECUDA, ETIMEOUT / EDEVICE (status
 * word set). */
K2T_API int k2t_msbfs(k2t_tree *t, int32_t dir, const uint32_t *sources, uint32_t B, int32_t *dist, void *work,
              uint32_t max_levels, uint32_t *levels, void *stream);

/* Bytes of the work buffer k2t_msbfs needs for this tree. */
K2T_API uint64_t k2t_msbfs_work_bytes(const k2t_tree *t);

/* Shape, per-level sizes and the device footprint broken down by part. */
K2T_API int k2t_stats_get(const k2t_tree *t, k2t_stats *s);

/* Signatures of one level as one byte per node (low 4 bits for k = 2 levels;
 * low 8 bits of the 16-bit signature in out[2i], high 8 bits in out[2i+1]
 * for k = 4 levels: the n_k4 top levels, and the leaf level of a tree with
 * leaf_k = 4).  cap is the capacity of out in bytes; *written is the
 * number of bytes the level needs.  ERANGE if cap is too small. */
K2T_API int k2t_level_signatures(const k2t_tree *t, uint32_t level, uint8_t *out, uint64_t cap,
                         uint64_t *written);

/* Device pointers of the uploaded image, for instrumentation: the signature
 * bytes of a level (nibble t of the level at byte t/2, low nibble first; the
 * 16-bit signature of node t at bytes 2t, 2t+1 for a leaf level with
 * leaf_k = 4) and its directory (NULL where absent). */
K2T_API int k2t_device_level(const k2t_tree *t, uint32_t level, const void **sig, const void **dir);

/* The cells of the matrix, decoded from the tree on the host, in level order
 * of their leaves.  ERANGE if cap < nnz (then *n_out = nnz). */
K2T_API int k2t_decode(const k2t_tree *t, uint32_t *rows, uint32_t *cols, uint64_t cap, uint64_t *n_out);

/* Release the tree, its host image and any library-owned device memory. */
K2T_API void k2t_free(k2t_tree *t);

K2T_API const char *k2t_strerror(int status);

/* The last CUDA error code seen by this thread inside the library (0 if none). */
K2T_API int k2t_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* K2T_H */
