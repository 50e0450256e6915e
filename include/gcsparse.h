/*
 * gcsparse.h -- C ABI of the grammar-compressed right-product engine.
 *
 * The method is the one of "Right Multiplication on Grammar-Compressed
 * Matrices: A Streaming, Memory-Bounded GPU Engine" (the pages):
 *   - a matrix M (n x m) is CSRV-encoded (Sec. 2 "CSRV", Eqs. 2.1-2.2): the
 *     distinct non-zero values form V, and each row becomes a string of
 *     terminals <l, j> (value V[l] in column j);
 *   - RePair compresses the row strings, never pairing across a row end, into
 *     rules N_i -> A_i B_i and a final sequence C (Sec. 2 "Grammar",
 *     Eqs. 2.3-2.4; Sec. 4.1);
 *   - levels (Eq. 3.1) and pass-through completion (Sec. 4.2) make the
 *     grammar properly layered (Def. 3.2), so that y = Mx is a bottom-up sweep
 *     in which level k reads only level k-1 (Lemma 3.3, Sec. 4.3);
 *   - the sweep needs only an associative combine, so the same schedule
 *     evaluates (+, x) in float32, 16 right-hand sides at once (Appendix A),
 *     exact int64, and the Boolean semiring on 64-bit bitsets (Sec. 5).
 *
 * Conventions
 *   - All indices are 0-based. Sizes are int64_t unless stated.
 *   - Every function returns a gc_status; none throws, exits or aborts.
 *     On failure gc_last_error() gives a message (thread-local).
 *   - Streams are cudaStream_t passed as void* (NULL = legacy default
 *     stream). Device work is enqueued on that stream and is asynchronous
 *     unless the entry point says it synchronises.
 *   - The library never allocates device memory for the product path: the
 *     caller allocates one device arena of gc_layout().arena_bytes and
 *     passes it to gc_upload(). Host objects (gc_grammar, gc_handle) are
 *     library-owned and released with the matching gc_free_*.
 */
#ifndef GCSPARSE_H
#define GCSPARSE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GC_OK = 0,
    GC_ERR_ARG = -1,              /* bad argument (null pointer, size, k, policy) */
    GC_ERR_OOM = -2,              /* host allocation failed                        */
    GC_ERR_CUDA = -3,             /* a CUDA runtime call failed                    */
    GC_ERR_INVALID_GRAMMAR = -4,  /* packed grammar failed validation              */
    GC_ERR_UNSUPPORTED = -5,      /* valid request this build cannot serve         */
    GC_ERR_TIMEOUT = -6,          /* a device-side wait ran out (status word)      */
    GC_ERR_NOT_CONVERGED = -7,    /* gc_reach hit max_iter before the fixpoint     */
    GC_ERR_IO = -8                /* gc_save / gc_load file error                  */
} gc_status;

/* Leaf / combine / emit policy of the sweep (Sec. 5: any monoid homomorphism).
 *   GC_F32_SUM       (+, x) in float32; k = 1, 4, 8, 16, 32, 64, 128 or 256
 *                    right-hand sides (Appendix A's batched product)
 *   GC_I64_SUM       (+, x) in exact int64; matrix values must be integers; k = 1
 *   GC_BOOL_OR       (OR, AND) on uint64 bitsets (64 sources per word); every
 *                    stored entry must be 1 (an edge); k = 1
 *   GC_F32_MIN_PLUS  tropical (min, +) in float32 (Sec. 5: one product is one
 *                    Bellman-Ford edge relaxation): y[i] = min over stored
 *                    M[i][j] of M[i][j] + x[j], each sum rounded to float32,
 *                    +inf for a row with no stored entry; min is exact, so y
 *                    is the same bit for bit whatever the order. x must hold
 *                    no NaN. k = 1 or k = 16                                 */
typedef enum { GC_F32_SUM = 0, GC_I64_SUM = 1, GC_BOOL_OR = 2, GC_F32_MIN_PLUS = 3 } gc_policy;

typedef struct {
    int64_t block_rows; /* 0: one grammar for all rows. >0: RePair runs on each
                           block of block_rows rows separately (Sec. 1 "row
                           blocks"); the blocks share one terminal table and
                           their levels are merged, so one sweep serves all.  */
    int32_t threads;    /* host threads for block-parallel RePair; 0 = all     */
    int32_t order;      /* within-level node order (any order is correct,
                           Sec. 4.3): 0 = by first column of the node's
                           expansion (locality of child reads, default);
                           1 = RePair creation order                          */
} gc_build_opts;

typedef struct {
    int64_t n, m, nnz;      /* matrix shape and stored non-zeros              */
    int64_t n_values;       /* |V|: distinct non-zero values                  */
    int64_t n_terminals;    /* alpha: distinct terminals <l, j>               */
    int64_t n_rules;        /* |R|: RePair nonterminals                       */
    int64_t n_pass;         /* pass-through nodes added by completion (+pt)   */
    int64_t n_nodes;        /* |R| + n_pass: layered nodes                    */
    int64_t depth;          /* L: number of levels                            */
    int64_t max_width;      /* w*: widest level = streaming-buffer length     */
    int64_t c_len;          /* |C| without row delimiters                     */
    int64_t n_roots;        /* rho: distinct nonterminals occurring in C      */
    int64_t n_blocks;       /* row blocks compressed separately (1 if none)   */
    double  repair_seconds; /* host time of CSRV + RePair                     */
    double  layer_seconds;  /* host time of levels + completion + packing     */
} gc_grammar_stats;

/* Arrays a built grammar can hand back (for checking and serialising).      */
typedef enum {
    GC_A_VALUES = 0,        /* float[n_values]: V ascending                              */
    GC_A_TERM_COL = 1,      /* int32[n_terminals]: column j of terminal t (sorted by j, l) */
    GC_A_TERM_VIDX = 2,     /* int32[n_terminals]: value index l of terminal t           */
    GC_A_RULES = 3,         /* int32[2*n_rules]: (A_i, B_i) per rule in creation order;
                               a child s >= 0 is N_s, s < 0 is terminal -s-1           */
    GC_A_C_OFF = 4,         /* int64[n+1]: row r's symbols are C[c_off[r]..c_off[r+1]) */
    GC_A_C_SYM = 5,         /* int32[c_len]: C in the GC_A_RULES symbol encoding        */
    GC_A_RULE_LEVEL = 6,    /* int32[n_rules]: Eq. 3.1 level of each rule               */
    GC_A_LVL_OFF = 7,       /* int64[depth+2]: level k's packed nodes are
                               [lvl_off[k], lvl_off[k+1]); lvl_off[0] = lvl_off[1] = 0 */
    GC_A_NODES = 8,         /* int32[2*n_nodes]: packed child references (a, b) per node;
                               c >= 0: slot c of level k-1's buffer; c < 0: T[-c-1]
                               where T[0] is the combine identity and T[p+1] leaf p.
                               A pass-through is (c, -1).                               */
    GC_A_LVL_ROOTS = 9,     /* int64[depth+2]: number of roots of level k; a level's
                               roots are its first nodes                                */
    GC_A_ROOT_OFF = 10,     /* int64[depth+2]: RV slot of level k's first root          */
    GC_A_C_REF = 11,        /* int32[c_len]: C packed: >= 0 RV slot, < 0 T[-c-1]         */
    GC_A_NODE_ID = 12       /* int32[n_nodes]: what each packed node is: rule i >= 0, or
                               -(u+1) for a pass-through carrying rule u                */
} gc_array;

typedef struct {
    int64_t arena_bytes;    /* total device bytes gc_upload needs (256-B aligned parts) */
    int64_t grammar_bytes;  /* read-only grammar arrays: nodes, level tables, leaves,
                               V-resolved leaf values, C offsets and references        */
    int64_t scratch_bytes;  /* T, root values RV, the two level buffers, status word   */
    int64_t staging_bytes;  /* device copies of x and y used by gc_matvec_host          */
    int64_t csr_bytes;      /* the same matrix as CSR: 4 B col + 4 B value per
                               non-zero + 4 (n+1) row pointers (8 (n+1) when
                               nnz >= 2^31), + x and y (Sec. 4.4 "Space")              */
} gc_arena_layout;

typedef struct gc_grammar gc_grammar;
typedef struct gc_handle gc_handle;
typedef struct gc_left_handle gc_left_handle;

/* Thread-local message of the last failure in this thread ("" if none).     */
const char* gc_last_error(void);

/* Library version string, e.g. "gcsparse 0.1 sm_103a".                     */
const char* gc_version(void);

/*
 * gc_build -- CSRV-encode, RePair-compress and layer a CSR matrix (host).
 * Sec. 2 (CSRV, RePair with row boundaries), Sec. 3 (Eq. 3.1), Sec. 4.1-4.3
 * (pass-through completion, level-major layout).
 *   row_ptr  int64[n+1], non-decreasing, row_ptr[0] = 0
 *   col      int32[nnz], in [0, m); a row's columns need not be sorted but
 *            must be distinct
 *   val      float[nnz], finite; NULL means every entry is 1. Zeros (+0/-0)
 *            are dropped, as CSRV stores non-zeros only. Values are the same
 *            V entry iff their float bit patterns are equal.
 *   opts     may be NULL (defaults: one block, all threads, locality order)
 *   out      receives a library-owned grammar; free with gc_free_grammar.
 * Host memory only; no device is touched. Errors: GC_ERR_ARG for bad CSR,
 * GC_ERR_OOM, GC_ERR_UNSUPPORTED when a count exceeds int32 limits.
 */
gc_status gc_build(int64_t n, int64_t m, const int64_t* row_ptr, const int32_t* col,
                   const float* val, const gc_build_opts* opts, gc_grammar** out);

/*
 * Streaming build in row blocks, for matrices too large to hand over as one
 * CSR (Sec. 1: row blocks compressed separately). gc_builder_add_rows
 * CSRV-encodes and RePair-compresses one block of rows [r0, r0 + rows) right
 * away and keeps only its grammar; it may be called concurrently from several
 * threads with different blocks. gc_builder_finish merges the blocks (one
 * value dictionary, one terminal table, rules numbered block after block)
 * and layers and packs the result like gc_build; it fails with GC_ERR_ARG
 * unless the blocks cover [0, n) exactly once. The block CSR follows the
 * gc_build rules with row_ptr[0] = 0. The builder is freed by
 * gc_builder_free (also after finish).
 */
typedef struct gc_builder gc_builder;
gc_status gc_builder_create(int64_t n, int64_t m, const gc_build_opts* opts, gc_builder** out);
gc_status gc_builder_add_rows(gc_builder* b, int64_t r0, int64_t rows, const int64_t* row_ptr,
                              const int32_t* col, const float* val);
gc_status gc_builder_finish(gc_builder* b, gc_grammar** out);
void gc_builder_free(gc_builder* b);

/*
 * gc_balance -- height balancing of a built grammar (Sec. 4.2 names
 * pre-balancing to a logarithmic height; Sec. 8 leaves it to future work).
 * The pages give no construction; this one rebuilds the rules bottom-up as an
 * AVL grammar: each rule becomes the join of its children's balanced forms,
 * so the two children of every rule differ in height by at most one and the
 * depth L is at most about 1.44 log2 of the longest expansion. Rules with the
 * same (left, right) pair are made once; rules C no longer reaches are
 * dropped. Expansions are unchanged, so products over the result equal the
 * original's. The result is layered and packed like gc_build's (default
 * order); *out is a new library-owned grammar (gc_free_grammar). Host memory
 * only. Errors: GC_ERR_ARG, GC_ERR_UNSUPPORTED (over 2^31-1 rules).
 */
gc_status gc_balance(const gc_grammar* g, gc_grammar** out);

/* Structural figures of a built grammar (Table 4.1's |R|, L, w*, +pt).      */
gc_status gc_stats(const gc_grammar* g, gc_grammar_stats* out);

/* Level widths w_1..w_L (Lemma 3.3; Sec. 4.2: width = live set).
 * w must hold cap >= depth entries.                                          */
gc_status gc_widths(const gc_grammar* g, int64_t* w, int64_t cap);

/* Size in bytes of an exported array (see gc_array).                        */
gc_status gc_export_size(const gc_grammar* g, gc_array which, int64_t* bytes);

/* Copy an array of the grammar into dst (host memory of dst_bytes bytes).   */
gc_status gc_export(const gc_grammar* g, gc_array which, void* dst, int64_t dst_bytes);

/*
 * gc_layout -- device bytes needed to serve products under a policy with up
 * to k_max right-hand sides (k_max one of GC_F32_SUM's widths above, 1 or 16
 * for GC_F32_MIN_PLUS, 1 otherwise). The level buffers hold k_max values a
 * node, so the scratch grows with k_max.
 * GC_ERR_UNSUPPORTED if the grammar's values do not fit the policy (non-
 * integer values for GC_I64_SUM, values other than 1 for GC_BOOL_OR).
 */
gc_status gc_layout(const gc_grammar* g, gc_policy policy, int32_t k_max, gc_arena_layout* out);

/*
 * gc_upload -- copy the packed grammar into a caller-owned device arena and
 * return a handle for products.
 *   arena        device pointer, 256-byte aligned, arena_bytes >= the
 *                gc_layout() figure for the same policy and k_max. It must
 *                outlive the handle; the library does not free it.
 *   stream       the copies are enqueued on it; the call returns after they
 *                are enqueued and the host-side validation (every child index
 *                within the level below, every terminal within alpha, every C
 *                reference within rho / alpha) has passed.
 * The handle keeps host copies of the level tables; the grammar may be freed
 * after the upload's copies completed (synchronise the stream first).
 * One product at a time per handle: the level buffers are shared by calls.
 */
gc_status gc_upload(const gc_grammar* g, gc_policy policy, int32_t k_max, void* arena,
                    int64_t arena_bytes, void* stream, gc_handle** out);

/*
 * gc_layout_ex / gc_upload_ex -- the same with the schedule chosen at upload:
 * GC_SCHED_PERSISTENT or GC_SCHED_PER_LEVEL (the layout of gc_layout /
 * gc_upload; the handle starts with that schedule), or GC_SCHED_DATAFLOW
 * (k_max = 1 only, else GC_ERR_UNSUPPORTED): the dataflow sweep's own layout
 * -- the levels cut into blocks with their dependency lists, three level
 * buffers, per-block ready flags -- on which the products run that schedule
 * (or its per-level launch sequence, GC_SCHED_PER_LEVEL). Its arena differs
 * from gc_layout's, so size it with gc_layout_ex and the same schedule. The
 * layout is the pages' level-synchronous sweep (Lemma 3.3) with the barrier
 * between levels replaced by per-block dependencies; on the 10,000 x 50,000
 * genotype grammar it measured slower than the persistent sweep (the latency
 * of a dependency hop exceeds that of a grid barrier there), so it is not
 * the default. Unknown schedules: GC_ERR_ARG.
 */
gc_status gc_layout_ex(const gc_grammar* g, gc_policy policy, int32_t k_max, int32_t schedule,
                       gc_arena_layout* out);
gc_status gc_upload_ex(const gc_grammar* g, gc_policy policy, int32_t k_max, int32_t schedule, void* arena,
                       int64_t arena_bytes, void* stream, gc_handle** out);

/*
 * gc_matvec -- y = M x on the device (Lemmas 2.1-2.2, Theorem 2.3, Sec. 4.3,
 * Appendix A for k > 1). Asynchronous on stream.
 *   x   device, m*k elements, row-major (x[j*k + c] is column j of input c)
 *       float for GC_F32_SUM and GC_F32_MIN_PLUS, int64_t for GC_I64_SUM,
 *       uint64_t for GC_BOOL_OR
 *   y   device, n*k elements, row-major, same element type; fully written
 *       (a row with no non-zeros gets the combine identity: 0, or +inf for
 *       GC_F32_MIN_PLUS)
 *   k   a width the policy supports, at most the handle's k_max (a k_max = 64
 *       handle also serves k = 1, 4, 8, 16, 32); x and y hold k values per
 *       column / row (4k bytes: k / 4 float4 lanes)
 * x and y must not overlap the arena. Deterministic: the same x gives the same
 * y bit for bit (fixed summation order, no atomics).
 * The device current at the call must be the one that was current at
 * gc_upload (the arena's device); otherwise GC_ERR_ARG. The same rule holds
 * for gc_matvec_host, gc_matvec_static, gc_reach and gc_sssp.
 */
gc_status gc_matvec(gc_handle* h, const void* x, void* y, int32_t k, void* stream);

/*
 * gc_matvec_host -- the same product with x and y in HOST memory: copies x
 * into the arena's staging area, runs gc_matvec, copies y back and
 * synchronises the stream before returning. Host buffers should be pinned
 * for full copy speed (pageable memory works but is slower).
 */
gc_status gc_matvec_host(gc_handle* h, const void* x_host, void* y_host, int32_t k,
                         void* stream);

/*
 * gc_reach -- Boolean-semiring fixpoint x <- x OR (M (x) x) from x0 until it
 * stops changing (Sec. 5; the pages stop at one pass and name the fixpoint as
 * the next step, Sec. 7 item 4). Requires GC_BOOL_OR and n == m.
 *   x0, x    device uint64_t[n]; bit b of x[i] ends set iff node i reaches a
 *            node whose bit b is set in x0. x may equal x0 (in place).
 *   iters    device int32_t[1]: products performed, the last of which changed
 *            nothing; -1 if max_iter was reached first.
 * Returns GC_ERR_NOT_CONVERGED (and records it in the status word, which
 * gc_check reports once) if max_iter products did not reach the fixpoint.
 * The loop runs on the device. Where the handle's product is one persistent
 * launch (the persistent schedule with the row or level emit: matrices with
 * short rows, such as graphs), the whole fixpoint is that one launch: each
 * product is followed, inside the kernel, by a grid barrier, the update
 * x = x OR y over the grid with a changed flag, and a second grid barrier
 * after which every CTA reads the flag; the call then synchronises the
 * stream once. Otherwise (the slice emit, the per-level and dataflow
 * schedules) products and update steps are enqueued in batches of 1, 2, 4,
 * 8, 8, ... with no host round trip inside a batch; the last update step to
 * finish records convergence, after which the kernels of the products
 * already enqueued return at once (x is unchanged by them). The host keeps
 * one batch enqueued ahead of the one whose convergence words it waits for
 * (an event on the stream), so the device does not idle between batches,
 * and returns once convergence (or max_iter) is known; the last batch's
 * early-return kernels and the iters write may still be on the stream:
 * synchronise it before reading x or iters on the host. Every later call on
 * the handle (products, gc_check, another fixpoint), on any stream, is
 * ordered after them. The first call pins 32 bytes of host memory and makes
 * three events, released by gc_free_handle. A grid barrier that times out
 * ends the call with GC_ERR_NOT_CONVERGED (iters -1) and leaves
 * GC_ERR_TIMEOUT in the status word for gc_check.
 */
gc_status gc_reach(gc_handle* h, const uint64_t* x0, uint64_t* x, int32_t max_iter,
                   int32_t* iters, void* stream);

/*
 * gc_update -- one fixpoint step on rows the caller holds: x[i] = x[i] OR y[i]
 * (GC_BOOL_OR, uint64_t) or x[i] = min(x[i], y[i]) (GC_F32_MIN_PLUS, float),
 * i < n, for a rank's share of a row-sharded fixpoint (Sec. 5's iteration,
 * rows split over GPUs: each rank updates its own rows, then the ranks gather
 * the new vector and agree on the changed flag).
 *   x, y     device arrays of n values (x updated in place; no overlap)
 *   changed  device int32_t[1]: set to 0, then to 1 if any element changed
 * Stream-ordered and asynchronous; no handle, no allocation. Errors:
 * GC_ERR_ARG (other policies, null pointers, n < 0), GC_ERR_CUDA.
 */
gc_status gc_update(gc_policy policy, void* x, const void* y, int64_t n, int32_t* changed, void* stream);

/*
 * gc_sssp -- tropical-semiring fixpoint x <- min(x, M (x) x) from x0 until it
 * stops changing: Bellman-Ford relaxation to the end (Sec. 5 measures one
 * pass, one edge relaxation, and names the iteration to the shortest-path
 * fixpoint as the next step, Sec. 7 item 4). Requires GC_F32_MIN_PLUS and
 * n == m; M[i][j] is the length of edge i -> j.
 *   x0, x    device float[n]; x[i] ends as min over nodes s of (length of a
 *            shortest path i -> s along out-edges) + x0[s], +inf if none
 *            (x0 = 0 at the sources, +inf elsewhere: distance to the nearest
 *            source). Sums round to float32 at every relaxation, so with
 *            non-integer lengths x is the float32 Bellman-Ford result, not
 *            the exact distance. x may equal x0 (in place). No negative cycle
 *            may be reachable: the iteration would not end before max_iter.
 *   iters    device int32_t[1]: products performed, the last of which changed
 *            nothing; -1 if max_iter was reached first.
 * Returns GC_ERR_NOT_CONVERGED (also recorded in the status word) if
 * max_iter products did not reach the fixpoint. The loop runs on the device
 * as described for gc_reach.
 */
gc_status gc_sssp(gc_handle* h, const float* x0, float* x, int32_t max_iter, int32_t* iters,
                  void* stream);

/* Synchronise the stream and return the device status word of the handle
 * (GC_OK, GC_ERR_TIMEOUT, GC_ERR_NOT_CONVERGED). The word is cleared after it
 * is read. While a GC_ERR_TIMEOUT is unread, products are skipped (y is not
 * written): a timed-out grid barrier leaves its counter part-way, and
 * gc_check restarts it.                                                     */
gc_status gc_check(gc_handle* h, void* stream);

/* Number of kernel launches the most recent gc_matvec on h enqueued.        */
gc_status gc_launch_count(const gc_handle* h, int64_t* launches);

/* Schedules of the sweep (the same values either way, bit for bit):
 *   GC_SCHED_PERSISTENT  one cooperative kernel per product, levels separated
 *                        by a grid barrier with bounded waits (default for
 *                        handles with k_max > 1; used when the device
 *                        supports cooperative launch)
 *   GC_SCHED_PER_LEVEL   one kernel per level plus the emit kernels, the
 *                        launch sequence of Listing 1 of the pages
 *   GC_SCHED_DATAFLOW    handles uploaded for it (gc_upload_ex): the levels
 *                        are cut into blocks of consecutive nodes; one
 *                        cooperative kernel stages each block's node pairs in
 *                        shared memory (a bulk copy) and starts the block once
 *                        the blocks that write its children have raised their
 *                        ready flags (bounded waits), so no grid barrier
 *                        separates the levels (Lemma 3.3's dependency, block by
 *                        block); the narrow top levels run as one block in
 *                        shared memory. Then the emit. On such a handle
 *                        GC_SCHED_PERSISTENT selects this schedule; on other
 *                        handles GC_SCHED_DATAFLOW is GC_ERR_UNSUPPORTED.      */
enum { GC_SCHED_PERSISTENT = 0, GC_SCHED_PER_LEVEL = 1, GC_SCHED_DATAFLOW = 2 };
gc_status gc_set_schedule(gc_handle* h, int32_t schedule);
/* The schedule products actually use (PER_LEVEL when cooperative launch is
 * unavailable).                                                             */
gc_status gc_get_schedule(const gc_handle* h, int32_t* schedule);

/*
 * gc_debug_inject -- failure injection for tests; never faults the GPU.
 *   what 0: normal operation. what 1: in the next persistent products, CTA 0
 *   skips its first grid-barrier arrival, so every other CTA's bounded wait
 *   runs out after timeout_cycles SM clock cycles; the kernel then sets the
 *   status word to GC_ERR_TIMEOUT and returns. gc_check reports it, clears
 *   it and resets the barrier state; products are skipped (y left unwritten)
 *   while a failure is unread.
 * timeout_cycles also sets the wait limit for what 0 (default 4e9 cycles).
 */
gc_status gc_debug_inject(gc_handle* h, int32_t what, int64_t timeout_cycles);

/*
 * gc_matvec_static -- y = M x without any device memory for scratch.
 * The pages have no counterpart; this is a library convenience. It serves
 * callers that cannot call cudaMalloc (or any allocator) where the product
 * runs: a process whose device memory is fully reserved up front, or code
 * that only receives input and output buffers. The product's scratch -- the
 * two level buffers, the tail buffer of the narrow top levels, the carry
 * slots, the emit's chunk or segment sums, the root values, the status word
 * and the grid-barrier counters -- lives in one fixed array compiled into the
 * library, of GC_STATIC_SCRATCH_BYTES bytes, that every GPU which loads the
 * library holds until the process exits. The handle's grammar (gc_upload) and
 * x are the inputs, y the output, as for gc_matvec; the handle's own scratch
 * is unused.
 *   Size limit: a product needs the sum of those parts for k values a node
 *   (each part rounded up to 256 bytes; about the handle's gc_layout
 *   scratch_bytes); a larger request returns GC_ERR_UNSUPPORTED with the
 *   sizes in gc_last_error().
 *   Set-up: the first call on a device, with that device current, looks up
 *   the array's device address (cudaGetSymbolAddress) once; make that first
 *   call before any stream capture.
 *   Sharing: every call uses the same array, which keeps the last call's
 *   contents; the call clears the status word and barrier counter itself.
 *   Calls that overlap on the GPU (other streams, other threads) race on it.
 *   Allocation: no cudaMalloc, cudaFree or allocating library routine.
 *   Returns after the product completed (it synchronises the stream), with
 *   GC_ERR_TIMEOUT if a device-side wait ran out.
 */
#define GC_STATIC_SCRATCH_BYTES (32ll << 20)
gc_status gc_matvec_static(gc_handle* h, const void* x, void* y, int32_t k, void* stream);

/*
 * Left product x^T = y^T M, i.e. x = M^T y (one right-hand side): the dual
 * of gc_matvec over the same grammar, under the same policies at k = 1:
 * GC_F32_SUM (float32), GC_I64_SUM (exact), GC_BOOL_OR (x[j] = OR of y[i]
 * over the entries (i, j): one forward step of a frontier) and
 * GC_F32_MIN_PLUS (x[j] = min of M[i][j] + y[i], float32, +inf for an
 * unused column: one forward Bellman-Ford relaxation). The pages name left
 * multiplication by pull-based reduction as future work (Sec. 8); here it is
 * a top-down sweep over the properly layered grammar in which every value is
 * a sum its reader gathers, in a fixed order (no atomics):
 *   RS[s]  = (+) of y[r] over row r's references to s in C (root slots and
 *            terminals),
 *   W[u]   = RS[u's slot] (roots) (+) the W of u's parents, level L first
 *            (every parent of a level-k node is at level k + 1, Def. 3.2),
 *   x[j]   = (+) over the terminals <l, j> of V[l] (x) (RS (+) the W of the
 *            nodes naming the terminal),
 * with (+) the policy's combine (sum, OR or min) and (x) its leaf map.
 * Long sums run over a warp with a fixed butterfly, so each is at most about
 * 64 + count / 32 + 5 additions deep. Deterministic: the same y gives the
 * same x bit for bit. Values: float, int64_t, uint64_t or float, by policy;
 * the policy's value checks are those of gc_layout (GC_ERR_UNSUPPORTED).
 *
 * gc_left_layout -- device bytes a left handle needs (grammar_bytes: the
 *   parent, seed and column lists and the task tables; scratch_bytes: RS, W,
 *   the terminal sums and the fixpoints' buffer and flag; staging_bytes 0; csr_bytes as in gc_layout for
 *   k = 1). Builds the plan on the host to size it.
 * gc_left_upload -- builds and checks the plan on the host (every reference
 *   within its list, every parent one level up, every segment in exactly one
 *   task), then copies it into a caller-owned arena (device, 256-byte
 *   aligned, at least arena_bytes, outliving the handle), enqueued on stream,
 *   and synchronises the stream. The grammar may be freed afterwards.
 * gc_left_matvec -- x = M^T y, asynchronous on stream: y device [n], x
 *   device [m] of the policy's type, fully written (a column no row uses gets
 *   the identity: 0, or +inf for GC_F32_MIN_PLUS). The L + 3
 *   steps (fewer when a step has nothing to sum) run as one CUDA graph of the
 *   handle, a chain of kernel nodes built by the first call; a call with new
 *   y or x pointers updates the two nodes that use them. One product at a
 *   time per handle, from one host thread (the graph and W are shared). x and
 *   y must not overlap the arena.
 * gc_left_launch_count -- kernels the last gc_left_matvec ran.
 * gc_free_left_handle -- host object and its graph; not the arena.
 */
gc_status gc_left_layout(const gc_grammar* g, gc_policy policy, gc_arena_layout* out);
gc_status gc_left_upload(const gc_grammar* g, gc_policy policy, void* arena, int64_t arena_bytes, void* stream,
                         gc_left_handle** out);
gc_status gc_left_matvec(gc_left_handle* h, const void* y, void* x, void* stream);
/*
 * gc_left_reach / gc_left_sssp -- the forward fixpoints with left products:
 * x <- x OR (M^T (x) x) (GC_BOOL_OR; bit b of x[j] ends set iff a node whose
 * bit b is set in x0 reaches j along out-edges, reflexively) and
 * x <- min(x, M^T (x) x) (GC_F32_MIN_PLUS; x[j] ends as the shortest path
 * length from a node s to j plus x0[s], minimised over s, float32 at every
 * relaxation). The reverse direction of gc_reach / gc_sssp (Sec. 5's BFS and
 * Bellman-Ford; the pages stop at one pass, Sec. 7 item 4). Requires n == m.
 *   x0, x    device uint64_t[n] / float[n]; x may equal x0 (in place).
 *   iters    device int32_t[1]: products performed, the last of which
 *            changed nothing; -1 if max_iter was reached first.
 * Returns GC_ERR_NOT_CONVERGED if max_iter products did not reach the
 * fixpoint. The loop runs on the device as described for gc_reach (batches,
 * one batch ahead, later calls ordered after the last batch); uses the
 * handle's graph and scratch (one call at a time per handle).
 */
gc_status gc_left_reach(gc_left_handle* h, const uint64_t* x0, uint64_t* x, int32_t max_iter, int32_t* iters,
                        void* stream);
gc_status gc_left_sssp(gc_left_handle* h, const float* x0, float* x, int32_t max_iter, int32_t* iters, void* stream);
gc_status gc_left_launch_count(const gc_left_handle* h, int64_t* launches);
void gc_free_left_handle(gc_left_handle* h);

/* Serialise / restore a built grammar (host file, little-endian, versioned). */
gc_status gc_save(const gc_grammar* g, const char* path);
gc_status gc_load(const char* path, gc_grammar** out);

void gc_free_grammar(gc_grammar* g);
void gc_free_handle(gc_handle* h);   /* host object only; not the arena */

#ifdef __cplusplus
}
#endif

#endif /* GCSPARSE_H */
