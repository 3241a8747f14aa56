/*
 * affinity.h -- C ABI of libaffinity, the GB300 (sm_103a) calibration pass
 * that scores head->neuron and neuron->next-layer-KV-group affinity for
 * affinity-aware sharding under Delayed Tensor Parallelism.
 *
 * Method: "Affinity-Aware Sharding for Delayed Tensor Parallelism"
 * (de Reynal, 2026), §3 "Method: affinity-aware layouts":
 *   - "Affinity scores": S_up in R^{G x I} (FO and ADD), S_down in R^{I x G},
 *     equation (5) for the first-order damage Delta_hk;
 *   - "Objective": unit-mass normalisation and J(h, nu), equation (6);
 *   - "Optimiser": scoring the G!/((G/L)!)^L labelled balanced partitions
 *     of the KV groups given the neighbouring neuron assignments.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  Tensors are dense, row-major, in PyTorch nn.Linear storage (out x in):
 *    a     [T, H*d_head]  attention output of every head; head h owns columns
 *                         h*d_head .. (h+1)*d_head-1
 *    x     [T, D]         residual entering the FFN's pre-norm
 *    Wo    [D, H*d_head]  attention output projection (W_o^(h) = its columns of head h)
 *    gamma [D]            FFN pre-norm gain
 *    Wg,Wu [I, D]         gate / up projections (row k = w^g_k, w^u_k)
 *    Wd    [D, I]         down projection (column k = w^d_k)
 *    gamma_next [D]       next layer's attention pre-norm gain
 *    Wq_next [H*d_head, D], Wk_next [G*d_head, D], Wv_next [G*d_head, D]
 *                         next layer's query / key / value projections
 *  Element type: dims->dtype (AFF_BF16 or AFF_FP32) for every tensor.
 *  Query head h belongs to KV group h / (H/G).
 *  Device pointers are caller-owned (e.g. allocated through PyTorch); the
 *  library never allocates, frees or keeps them.  Inputs are read-only.
 *  Every device pointer must be 16-byte aligned.
 *  Outputs are overwritten, never accumulated into.
 *  All device work is enqueued on `stream` in order; no call synchronises
 *  the device or the stream.  A call returns AFF_OK once its work is
 *  enqueued; errors found on the device are latched into a status word in
 *  the workspace and read with affinity_device_status().
 *  Validation happens before any launch: a call that returns an error code
 *  other than AFF_ERR_CUDA has enqueued nothing.
 *  For fixed inputs, shapes and library build the outputs are bit-identical
 *  from run to run (fixed reduction orders, no floating-point atomics).
 *
 *  bf16 path numerics: tensor-core operands are staged as fp16 (the
 *  normalised FFN input gamma*x/r, a/r, the gate/up weights, the folded
 *  per-head matrices) and contracted with fp32 accumulation; the SwiGLU
 *  operating point stays fp32; token sums are finished in fp64.  Each staged
 *  tensor is multiplied by a power of two chosen on the device from its
 *  largest magnitude (or a bound on it) and the fp32 results by the inverse,
 *  so affinity_up accepts every finite bf16 input: values far outside fp16's
 *  range (|v| < 65504, normal above 2^-14) give the same scores as in range,
 *  with the rescaling limited to factors 2^-60 .. 2^60 per tensor.  A
 *  non-finite input latches AFF_ERR_RANGE.  affinity_down stages without
 *  rescaling its down-projection side (alpha, W_d, the next layer's q/k/v
 *  rows): there an fp16 overflow latches AFF_ERR_RANGE.  fp32 path: fp32
 *  arithmetic on the CUDA cores (meant for small shapes).
 */
#ifndef AFFINITY_H
#define AFFINITY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define AFF_API __attribute__((visibility("default")))
#else
#define AFF_API
#endif

/* Same type as cudaStream_t / CUstream; NULL is the legacy default stream. */
typedef struct CUstream_st* aff_stream_t;

typedef enum {
  AFF_OK = 0,
  AFF_ERR_INVALID_ARG = 1,        /* NULL pointer, bad enum, non-positive size */
  AFF_ERR_UNSUPPORTED_SHAPE = 2,  /* shape outside the constraints listed below */
  AFF_ERR_UNSUPPORTED_DTYPE = 3,
  AFF_ERR_ARCH = 4,               /* current device is not sm_103 / no device */
  AFF_ERR_WORKSPACE = 5,          /* workspace NULL, too small or misaligned */
  AFF_ERR_CUDA = 6,               /* a CUDA call failed; see affinity_last_cuda_error() */
  AFF_ERR_DEVICE_TIMEOUT = 7,     /* a kernel's bounded wait expired (device-latched) */
  AFF_ERR_RANGE = 8,              /* a non-finite input, or an fp16 overflow where nothing rescales (device-latched) */
  AFF_ERR_ALIGNMENT = 9,          /* a pointer is not 16-byte aligned */
  AFF_ERR_NO_CONVERGENCE = 10     /* an iterative solver hit its iteration cap (device-latched) */
} aff_status;

typedef enum {
  AFF_MODE_FO = 0,   /* S_hk = E_t[Delta_hk^2] * ||w^d_k||^2, Delta from eq. (5) */
  AFF_MODE_ADD = 1,  /* S_hk = E_t[(p_h.w^g_k)^2 + (p_h.w^u_k)^2] */
  AFF_MODE_LOO = 2   /* S_hk = E_t[(g_k - g_k^(-h))^2 + (u_k - u_k^(-h))^2]: exact leave-one-out,
                        the pre-activations recomputed from x - a_h W_o^(h) with its own rms
                        (AFF_BF16 only) */
} aff_mode;

typedef enum { AFF_BF16 = 0, AFF_FP32 = 1 } aff_dtype;

/*
 * aff_dims.flags bits.
 *   AFF_FLAG_ADD_DIRECT: ADD mode contracts every token with every folded
 *     neuron row (T x 2I x d_head multiply-adds per head).  Without it, AFF_BF16
 *     ADD with d_head <= 128 takes the second-moment form: per head the d_head x
 *     d_head matrix C_h = sum_t (a_h/r)(a_h/r)^T on the tensor cores, then
 *     m^T C_h m for every folded row m -- the same sum in a different rounding
 *     order (E_t[(p_h.w)^2] = m^T E_t[a~ a~^T] m).  Other modes ignore the bit.
 */
#define AFF_FLAG_ADD_DIRECT 1u

/*
 * Layer shape.  T tokens, model width D, H query heads in G KV groups of
 * H/G heads, head width d_head, I FFN neurons; eps is the rms epsilon
 * (r = sqrt(mean_d x_d^2 + eps)); dtype an aff_dtype; flags 0 or AFF_FLAG_ADD_DIRECT
 * (any other bit is AFF_ERR_INVALID_ARG).
 *
 * Constraints: all sizes >= 1, H % G == 0.  AFF_BF16 additionally needs
 * D % 8 == 0, d_head % 8 == 0 and I % 8 == 0 (16-byte row strides for the
 * tensor-memory copies); any T >= 1 (a ragged last token tile is handled).
 * AFF_FP32 has no further constraint.  eps must be finite and >= 0.
 */
typedef struct {
  int64_t T, D, H, G, d_head, I;
  float eps;
  int32_t dtype;
  uint32_t flags;
} aff_dims;

/*
 * Bytes of device workspace that affinity_up (down == 0) or affinity_down
 * (down != 0) needs for this shape and mode (mode is ignored when down != 0).
 * For AFF_MODE_ADD the size also depends on dims->flags (AFF_FLAG_ADD_DIRECT
 * selects the direct form, whose per-chunk partial sums are larger).
 * The workspace must be 256-byte aligned.  Returns AFF_ERR_INVALID_ARG /
 * AFF_ERR_UNSUPPORTED_SHAPE / AFF_ERR_UNSUPPORTED_DTYPE for bad dims.
 */
AFF_API aff_status affinity_workspace_size(const aff_dims* dims, int32_t mode, int32_t down, size_t* bytes);

/*
 * S_up for one layer ("Affinity scores", §3; equation (5)).
 *   FO : S_up[g, k] = sum_{h in g} E_t[Delta_hk^2] * ||w^d_k||^2
 *        Delta_hk = silu'(g_k) u_k (p_h.w^g_k) + silu(g_k) (p_h.w^u_k),
 *        p_h = gamma * (a_h W_o^(h)) / r,  r = rms(x),
 *        g_k = (gamma*x/r).w^g_k,  u_k = (gamma*x/r).w^u_k.
 *   ADD: S_up[g, k] = sum_{h in g} E_t[(p_h.w^g_k)^2 + (p_h.w^u_k)^2].
 *   LOO: S_up[g, k] = sum_{h in g} E_t[(g_k - g_k^(-h))^2 + (u_k - u_k^(-h))^2] with
 *        g_k^(-h) = (gamma*(x - c_h)/rms(x - c_h)).w^g_k, c_h = a_h W_o^(h) (likewise u):
 *        the exact leave-one-out change ("Affinity scores": it differs from ADD
 *        only by the rms change).  Computed as g (1 - rho) + rho (p_h.w^g) with
 *        rho = r / rms(x - c_h) from a tensor-core pass over c_h / r.  AFF_BF16
 *        only (AFF_ERR_UNSUPPORTED_DTYPE for AFF_FP32).
 * E_t is the mean over the T tokens.  Wd is read only in FO mode (it may be
 * NULL in ADD mode).
 * Outputs (device, fp32): S_out [G, I] row-major; S_head_out [H, I] (the
 * per-query-head scores before the group sum) or NULL.
 * workspace: device, >= affinity_workspace_size(dims, mode, 0) bytes,
 * 256-byte aligned; its contents are scratch (no state between calls except
 * the status word); two calls must not use one workspace concurrently.
 */
AFF_API aff_status affinity_up(const void* a, const void* x, const void* Wo, const void* gamma,
                       const void* Wg, const void* Wu, const void* Wd,
                       const aff_dims* dims, int32_t mode,
                       float* S_out, float* S_head_out,
                       void* workspace, size_t workspace_bytes, aff_stream_t stream);

/*
 * affinity_up without a workspace argument.  The paper has no counterpart:
 * this entry point serves callers that cannot allocate device memory --
 * for example a plugin hosted by a framework that owns every device
 * allocation and hands plugins no scratch, or a process whose memory pool
 * has already reserved the whole device.  It computes exactly what
 * affinity_up computes (same arguments minus the workspace) and calls no
 * allocator; its scratch is one 64 MiB array compiled into the library,
 * which every GPU that loads the library holds until the process exits.
 *   - Shapes whose affinity_workspace_size(dims, mode, 0) exceeds 64 MiB
 *     (67108864 bytes) are refused with AFF_ERR_WORKSPACE; nothing is
 *     enqueued.
 *   - The first call on a device looks up the array's device address (once
 *     per device, with that device current); make that first call before
 *     any stream capture.  Under CUDA's lazy module loading (the default)
 *     that lookup is also when the 64 MiB is reserved on the device, not
 *     when the library is loaded: a caller whose pool is about to take the
 *     whole device must make its first call (or one
 *     affinity_static_device_status call) before the pool reserves it;
 *     otherwise the reservation fails and the call returns AFF_ERR_CUDA.
 *   - All calls share the one array, which keeps the last call's contents
 *     (each call writes every part it reads).  Calls whose work overlaps on
 *     the GPU -- on different streams, or from different host threads --
 *     race on it: serialise them.  The device status word lives in the
 *     array too: read it with affinity_static_device_status(), not
 *     affinity_device_status().
 */
AFF_API aff_status affinity_up_static(const void* a, const void* x, const void* Wo, const void* gamma,
                              const void* Wg, const void* Wu, const void* Wd,
                              const aff_dims* dims, int32_t mode,
                              float* S_out, float* S_head_out, aff_stream_t stream);

/*
 * The status word of affinity_up_static's array: synchronises `stream`, then
 * reads and clears what the kernels of the previous affinity_up_static call
 * on the current device latched (AFF_ERR_DEVICE_TIMEOUT, AFF_ERR_RANGE);
 * returns AFF_OK if none was set.  Like affinity_device_status, but for the
 * array that stands in for the workspace; it allocates nothing either.  The
 * paper has no counterpart.
 */
AFF_API aff_status affinity_static_device_status(aff_stream_t stream);

/*
 * S_down for one layer ("Affinity scores", §3, down edge):
 *   S_down[k, g] = E_t[alpha_k^2 / r'^2] * ||b_gk||^2,
 *   alpha_k = silu(g_k) u_k,  b_gk = W^qkv_g (gamma_next * w^d_k),
 *   W^qkv_g = [query rows of g's H/G heads; key rows of g; value rows of g],
 *   r' = rms(x') with x' = x + sum_k alpha_k w^d_k (the residual after this
 *   FFN, which is the next attention's pre-norm input) and the same eps.
 * Output S_out [I, G] row-major fp32 (device).  Workspace as for affinity_up
 * with down != 0.
 */
AFF_API aff_status affinity_down(const void* x, const void* gamma, const void* Wg, const void* Wu,
                         const void* Wd, const void* gamma_next, const void* Wq_next,
                         const void* Wk_next, const void* Wv_next,
                         const aff_dims* dims, float* S_out,
                         void* workspace, size_t workspace_bytes, aff_stream_t stream);

/*
 * Synchronises `stream`, then reads and clears the status word that kernels
 * of the previous affinity_up / affinity_down call on this workspace latch
 * (AFF_ERR_DEVICE_TIMEOUT; AFF_ERR_RANGE for a non-finite input, or an fp16
 * overflow on affinity_down's unscaled side); returns AFF_OK if none was set.
 */
AFF_API aff_status affinity_device_status(void* workspace, aff_stream_t stream);

/*
 * Self-test of the device-side failure path (no counterpart in the paper).
 * Every pipeline wait inside the library's kernels is bounded: past its time
 * limit it latches AFF_ERR_DEVICE_TIMEOUT in the workspace status word and
 * returns instead of spinning, so the context stays usable.  This call
 * launches one kernel whose single wait can never be satisfied, with the
 * given limit; afterwards affinity_device_status(workspace) must report
 * AFF_ERR_DEVICE_TIMEOUT.  Nothing faults, traps or hangs.
 *   workspace  device, >= 256 bytes, 256-byte aligned (its status word is
 *              cleared first)
 *   limit_ns   1e3 .. 1e10
 */
AFF_API aff_status affinity_selftest_timeout(void* workspace, size_t workspace_bytes, int64_t limit_ns,
                                             aff_stream_t stream);

/*
 * Host-only helper ("Optimiser", §3): score every labelled balanced
 * partition h of G KV groups onto L devices (G/L groups per device) by
 * sum_g C[g, h(g)], where C [G, L] (host, row-major, fp64) is the gain of
 * putting group g on device l.  Partitions are enumerated in lexicographic
 * order of (h(0), ..., h(G-1)); the first maximum wins ties.
 *   scores      host [count] or NULL
 *   count       number of partitions, G! / ((G/L)!)^L (2520 for G=8, L=4)
 *   best_index  index of the best partition in that order
 *   best_assign host [G]: the best partition's device of each group, or NULL
 * Requires 1 <= L <= G <= 16 and G % L == 0 (AFF_ERR_INVALID_ARG otherwise)
 * and at most 1e8 partitions (AFF_ERR_UNSUPPORTED_SHAPE otherwise); when
 * scores != NULL the caller must size it with a first call that passes
 * scores == NULL.
 */
AFF_API aff_status affinity_score_partitions(const double* C, int32_t G, int32_t L, double* scores,
                                     int64_t* count, int64_t* best_index, int32_t* best_assign);

/*
 * Host-only helper ("Optimiser", §3): the gain C [G, L] (fp64) of placing
 * group g of layer i on device l given the neuron maps, from unit-mass
 * matrices:  C[g, l] = sum_{k: nu_i(k) = l} Shat_up_i[g, k]
 *                    + sum_{k: nu_prev(k) = l} Shat_down_prev[k, g].
 * Shat_up_i [G, I], Shat_down_prev [I, G] (NULL for the first layer),
 * nu_i / nu_prev [I] device indices in [0, L).  All host memory.
 */
AFF_API aff_status affinity_group_gain(const double* Shat_up_i, const int32_t* nu_i,
                               const double* Shat_down_prev, const int32_t* nu_prev,
                               int32_t G, int64_t I, int32_t L, double* C);

/*
 * Host-only helper ("Objective", equation (6)): total co-located affinity
 *   J = sum_i sum_{g,k: h_i(g) = nu_i(k)} Shat_up_i[g, k]
 *     + sum_{i < N-1} sum_{k,g: nu_i(k) = h_{i+1}(g)} Shat_down_i[k, g]
 * for N layers.  Shat_up: N contiguous [G, I] fp64 blocks; Shat_down: N-1
 * contiguous [I, G] blocks (may be NULL when N == 1); h: N x [G];
 * nu: N x [I]; all host memory.
 */
AFF_API aff_status affinity_objective(const double* Shat_up, const double* Shat_down,
                              const int32_t* h, const int32_t* nu,
                              int32_t N, int32_t G, int64_t I, double* J);

/*
 * Host-only helper ("Objective", §3: each affinity matrix is normalised to
 * unit mass before it enters J): out[i] = S[i] / sum_j S[j], summed in fp64
 * in index order.  S: host fp32 [n] (an S_up [G, I] or S_down [I, G] as
 * written by affinity_up / affinity_down); out: host fp64 [n].
 * AFF_ERR_INVALID_ARG if n < 1 or the sum is not positive and finite.
 */
AFF_API aff_status affinity_unit_mass(const float* S, int64_t n, double* out);

/*
 * Host-only helper ("Optimiser", §3, the head step of the alternating
 * search): with the neuron maps nu of all N layers fixed, choose for every
 * layer i the balanced KV-group map h_i that maximises its gain
 * C_i = affinity_group_gain(Shat_up_i, nu_i, Shat_down_{i-1}, nu_{i-1}), by
 * scoring every balanced partition (affinity_score_partitions, first
 * maximum on ties).  Because h_i enters J (equation (6)) only through layer
 * i's up term and layer i-1's down term, the result maximises J over all h
 * for the given nu.
 *   Shat_up   host fp64, N contiguous [G, I] unit-mass blocks
 *   Shat_down host fp64, N-1 contiguous [I, G] blocks (may be NULL if N == 1)
 *   nu        host int32 N x [I], values in [0, L)
 *   h_out     host int32 N x [G] (written)
 *   J_out     host fp64: J of (h_out, nu), or NULL
 * Same limits on (G, L) as affinity_score_partitions.
 */
AFF_API aff_status affinity_best_heads(const double* Shat_up, const double* Shat_down,
                                       const int32_t* nu, int32_t N, int32_t G, int64_t I,
                                       int32_t L, int32_t* h_out, double* J_out);

/*
 * Host-only helper for token-sharded calibration (one GPU per shard of the
 * calibration tokens).  Every entry of S_up, S_head and S_down is a mean over
 * tokens times a per-neuron factor (§3 "Affinity scores": E_t[...]), so the
 * full-set value is the token-weighted mean of the shards' values:
 *   out[j] = sum_r T_r * S_r[j] / sum_r T_r,
 * accumulated in fp64 in shard order r = 0, 1, ... (deterministic).
 *   S_shards  n_shards host pointers to fp32 [n] (may be NULL where T_r == 0)
 *   T_shards  host int64 [n_shards], tokens of each shard, >= 0, sum > 0
 *   out       host fp32 [n]; may alias none of the inputs
 */
AFF_API aff_status affinity_combine_shards(const float* const* S_shards, const int64_t* T_shards,
                                           int32_t n_shards, int64_t n, float* out);

/* ------------------------------------------------------------------------
 * Layout search ("Optimiser", §3).  Unit-mass matrices are fp64.
 * ---------------------------------------------------------------------- */

/* Options of the neuron solver; zero fields take the defaults. */
typedef struct {
  int32_t dual_iters;   /* dual-ascent iterations on the device offsets (default 300) */
  double dual_decay;    /* step decay per iteration, in (0, 1] (default 0.98) */
  int64_t max_cycles;   /* cap on applied exchange cycles (default 64 * I) */
} aff_assign_opts;

/*
 * The gain of putting neuron k of layer i on device l, on the GPU:
 *   M[k, l] = sum_{g: h_i(g) = l} Shat_up_i[g, k]
 *           + sum_{g: h_next(g) = l} Shat_down_i[k, g]
 * (the second sum only when Shat_down_i is given; the last layer of a stack
 * has none).  Groups are added in ascending order, up term first.
 *   Shat_up_i   device fp64 [G, I];  Shat_down_i device fp64 [I, G] or NULL
 *   h_i, h_next host int32 [G], devices in [0, L) (h_next NULL iff Shat_down_i is)
 *   M_out       device fp64 [I, L]
 * 1 <= G <= 16, 1 <= L <= 8; 8-byte aligned device pointers.  Enqueued on
 * `stream`; nothing is synchronised.
 */
AFF_API aff_status affinity_neuron_gain(const double* Shat_up_i, const double* Shat_down_i,
                                        const int32_t* h_i, const int32_t* h_next, int32_t G, int64_t I,
                                        int32_t L, double* M_out, aff_stream_t stream);

/*
 * Best balanced neuron map of each of `n_layers` independent problems: nu
 * maximises sum_k M[k, nu(k)] with exactly I/L neurons per device.  One CTA
 * per problem runs dual ascent on the L device offsets, a fix-up that makes
 * single cheapest moves from over- to under-full devices, and then applies
 * the best exchange cycle of devices (one neuron moved out of each device on
 * the cycle, the best neuron per ordered device pair) while one gains more
 * than rounding.  When none gains, the map is optimal, so the value equals
 * the Hungarian solution up to rounding; ties between equally good maps are
 * broken by the fixed search order.
 *   M          device fp64 [n_layers][I][L]
 *   nu_out     device int32 [n_layers][I]
 *   value_out  device fp64 [n_layers]: sum_k M[k, nu(k)]
 *   workspace  device, >= 256 B, 256-byte aligned (status word; read it with
 *              affinity_device_status: AFF_ERR_NO_CONVERGENCE if max_cycles
 *              was reached, the map then being balanced but not proven best)
 * Requires 1 <= L <= 8, I % L == 0, L <= I <= 49152.  Deterministic.
 */
AFF_API aff_status affinity_assign_neurons(const double* M, int32_t n_layers, int64_t I, int32_t L,
                                           const aff_assign_opts* opts, int32_t* nu_out,
                                           double* value_out, void* workspace, size_t workspace_bytes,
                                           aff_stream_t stream);

/* Options of the alternating search; zero fields take the defaults. */
typedef struct {
  int32_t max_sweeps;          /* sweeps of (neuron step, head step) at most (default 16) */
  int32_t freeze_heads;        /* nonzero: keep every h_i as given */
  int32_t freeze_neurons;      /* nonzero: keep every nu_i as given */
  int32_t minimise;            /* nonzero: minimise J instead of maximising it */
  const uint8_t* layer_mask;   /* host [N]: 0 keeps layer i's maps as given; NULL: all move */
  aff_assign_opts assign;      /* neuron-solver options */
} aff_layout_opts;

/* Device workspace bytes for affinity_optimise_layout. */
AFF_API aff_status affinity_layout_workspace_size(int32_t N, int32_t G, int64_t I, int32_t L,
                                                  size_t* bytes);

/*
 * Alternating maximisation of J (equation (6)) over balanced layouts of an
 * N-layer stack ("Optimiser", §3).  From the given maps, each sweep first
 * sets every layer's neuron map to the best one given h_i and h_{i+1} (GPU,
 * affinity_neuron_gain + affinity_assign_neurons over all layers at once),
 * then every layer's KV-group map to the best balanced partition given
 * nu_{i-1} and nu_i (host, affinity_group_gain + affinity_score_partitions).
 * Each step is optimal given the rest, so J never decreases; the search
 * stops when a sweep gains less than 1e-12 relative, or after max_sweeps.
 *   Shat_up   host fp64, N contiguous [G, I] unit-mass blocks
 *   Shat_down host fp64, N-1 contiguous [I, G] blocks (NULL if N == 1)
 *   h, nu     host int32 N x [G] and N x [I]: the balanced starting maps on
 *             entry (e.g. contiguous), the result on return
 *   J_out     host fp64: J of the result;  sweeps_out: sweeps run (may be NULL)
 * G % L == 0, G <= 16 and the limits of affinity_assign_neurons.
 * Synchronises `stream` once per sweep (the head step runs on the host).
 */
AFF_API aff_status affinity_optimise_layout(const double* Shat_up, const double* Shat_down, int32_t N,
                                            int32_t G, int64_t I, int32_t L, const aff_layout_opts* opts,
                                            int32_t* h, int32_t* nu, double* J_out, int32_t* sweeps_out,
                                            void* workspace, size_t workspace_bytes, aff_stream_t stream);

/* ------------------------------------------------------------------------
 * Layout realisation ("The layout as a free variable", §3).
 * ---------------------------------------------------------------------- */

/*
 * Host-only: the storage orders that realise a balanced layout.  KV groups
 * and neurons are sorted by device, stably (ascending index within a
 * device); every group brings its H/G query heads in ascending order.
 *   h [G], nu [I]: devices in [0, L), G/L groups and I/L neurons per device
 *   group_order [G], head_order [H], neuron_order [I]: written; position p
 *   of the permuted storage holds original group / head / neuron order[p],
 *   and device l's shard is positions [l*n/L, (l+1)*n/L).
 * The permuted weights are then (rows of a matrix stored out x in):
 *   Wq rows by head_order (blocks of d_head rows), Wk/Wv rows by
 *   group_order (blocks of d_head rows), Wo columns by head_order (blocks of
 *   d_head columns), Wg/Wu rows by neuron_order, Wd columns by neuron_order;
 *   see affinity_gather_blocks.
 */
AFF_API aff_status affinity_layout_orders(const int32_t* h, const int32_t* nu, int32_t G, int64_t H,
                                          int64_t I, int32_t L, int32_t* group_order, int32_t* head_order,
                                          int32_t* neuron_order);

/*
 * Device gather of fixed-size blocks: out[r][j] = in[r][order[j]] for
 * r < rows, j < n_blocks, each block `block_bytes` bytes and each row
 * n_blocks * block_bytes bytes (contiguous).  A row permutation of a matrix
 * is rows = 1 with one or more matrix rows per block; a column permutation
 * is rows = the matrix's row count with one or more columns per block.
 *   in, out    device, non-overlapping; any alignment (wider words are used
 *              when pointers and block size allow)
 *   order      HOST int32 [n_blocks], a permutation of 0..n_blocks-1
 *              (AFF_ERR_INVALID_ARG otherwise; checked before any launch)
 *   workspace  device, >= 4 * n_blocks bytes, 256-byte aligned: the order
 *              is copied there on `stream`.  From pageable memory the copy is
 *              staged before the call returns; a pinned `order` must stay
 *              valid until the stream has run the copy.
 * Bit-exact data movement; enqueued on `stream`.
 */
AFF_API aff_status affinity_gather_blocks(const void* in, void* out, int64_t rows, int64_t n_blocks,
                                          int64_t block_bytes, const int32_t* order, void* workspace,
                                          size_t workspace_bytes, aff_stream_t stream);

/*
 * Profiling hook (no effect on results): register two caller-created CUDA
 * events (cudaEvent_t handles) that later affinity_up / affinity_down calls
 * made from this host thread record on their stream immediately before and
 * after their dominant tensor-core kernel -- the operating point + per-head
 * contraction kernel for affinity_up, the gate/up (alpha) kernel for
 * affinity_down.  Pass two NULLs to stop recording.  The events must outlive
 * the calls that record them.
 */
AFF_API aff_status affinity_set_timing_events(void* start_event, void* stop_event);

/* Static text for a status code. */
AFF_API const char* affinity_strerror(aff_status status);

/* Text of the last CUDA error seen by this thread (empty if none). */
AFF_API const char* affinity_last_cuda_error(void);

/* ABI version: major * 10000 + minor * 100 + patch. */
AFF_API int32_t affinity_version(void);

#ifdef __cplusplus
}
#endif

#endif /* AFFINITY_H */
