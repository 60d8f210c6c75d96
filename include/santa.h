/*
 * santa.h — C ABI of libsanta.so: SANTA++ decode-step attention on one GB300 (sm_103a).
 *
 * Sources of the method (cited by page title and section):
 *   [ABS]  "SANTA++: Sampling Attention through Representative Keys" (arXiv 2609.35629),
 *          abstract, as printed on arxivdaily.com and fugumt.com.
 *   [EXP]  "SANTA++：用代表性 Key 采样把 KV cache 读带宽砍掉 80%" (papers.ananclaw.com
 *          explainer), section 三 (the core method), its five-step pipeline and 3.1.
 *
 * What the library computes, for every sequence b and KV head h (a "unit"):
 *   teams      the n = ceil(seq_len/T) contiguous blocks of T cached tokens; team i is the
 *              KV page page_table[b][i].                                   [ABS; EXP step 1]
 *   reps       rep_i = mean of team i's valid keys (fp32 side buffer).     [ABS; EXP step 2]
 *   probs      s_{g,i} = q_g . rep_i / sqrt(d) for the G = Hq/Hkv query heads g of the group;
 *              p_{g,i} = softmax_i(s_{g,.});  p_i = (1/G) sum_g p_{g,i}.   [ABS; EXP step 2]
 *   sampling   M i.i.d. draws with replacement from p; draw r uses Philox4x32-10 (Salmon et
 *              al., SC'11) with key (lo32(seed), hi32(seed)) and counter (r, h, b, 0); word 0
 *              x gives u = (x + 0.5) 2^-32, and the draw is the smallest i with u*Z < C_i,
 *              C the running sum of p and Z = C_{n-1}.  S = the distinct drawn teams,
 *              ascending; pi_i = 1 - (1 - p_i)^M.                          [ABS; EXP step 3]
 *   attention  for each query head g of the group, the Horvitz-Thompson ratio
 *              out_g = sum_{i in S} (1/pi_i) sum_{j in team i} e^{s_j} v_j
 *                    / sum_{i in S} (1/pi_i) sum_{j in team i} e^{s_j},
 *              s_j = q_g . k_j / sqrt(d).                               [ABS; EXP steps 4-5]
 *
 * Layouts (all row-major, all device memory unless stated):
 *   q          [B][Hq][d]        dtype; query head hq reads KV head hq / G.
 *   k_pool     [P][Hkv][T][d]    dtype; page p, head h is one contiguous T*d block.
 *   v_pool     [P][Hkv][T][d]    dtype.
 *   reps       [P][Hkv][d]       fp32.
 *   page_table [B][max_teams]    int32, physical page of team i of sequence b.
 *   seq_lens   [B]               int32, 1 <= seq_len <= max_teams*T.
 *   out        [B][Hq][d]        fp32.
 *   draw_ids   [B][Hkv][M]       int32, team index of every draw, in draw order.
 *   sel_ids    [B][Hkv][M]       int32, S ascending, padded with -1.
 *   sel_count  [B][Hkv]          int32, |S|.
 *   pi         [B][Hkv][M]       fp32, pi_i aligned with sel_ids, padded with 0.
 *   team_probs [B][Hkv][max_teams] fp32 (optional), p_i, padded with 0.
 *
 * Conventions:
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy default stream)
 *     and runs on the device that is current on the calling thread.
 *   - The caller owns and allocates every buffer.  The library allocates no memory and keeps
 *     no per-call state; calls on different streams with disjoint buffers may overlap.
 *   - Host-side argument errors return SANTA_ERR_INVALID_ARG / SANTA_ERR_UNSUPPORTED and
 *     launch nothing.  A failed launch returns SANTA_ERR_CUDA.
 *   - Errors only visible on the device (an out-of-range page id or seq_len) never trap:
 *     the kernel ORs a SANTA_DEV_* bit into *device_status, skips the offending team or
 *     unit (a skipped unit gets out = 0 and sel_count = 0) and carries on.  The caller
 *     zeroes *device_status, synchronises and reads it; a non-zero word means the outputs
 *     of the affected units are not meaningful (SANTA_ERR_DEVICE_STATUS).
 *   - Supported shapes: dtype f32 or bf16; head_dim 64 or 128; team_size 64 or 128;
 *     1 <= G <= 8; 1 <= M <= 4096; max_teams <= 16384.  All pointers 16-byte aligned.
 */
#ifndef SANTA_H
#define SANTA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SANTA_ABI_VERSION 1

typedef enum santa_status {
  SANTA_OK = 0,
  SANTA_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misaligned pointer, short workspace */
  SANTA_ERR_UNSUPPORTED = 2,   /* a shape outside the supported set above */
  SANTA_ERR_CUDA = 3,          /* a CUDA runtime call or kernel launch failed */
  SANTA_ERR_DEVICE_STATUS = 4, /* reserved for callers: *device_status was non-zero */
  SANTA_ERR_SCRATCH_LIMIT = 5  /* santa_decode_noalloc: the problem needs more scratch than
                                  santa_noalloc_scratch_bytes() */
} santa_status;

typedef enum santa_dtype { SANTA_F32 = 0, SANTA_BF16 = 1 } santa_dtype;

/* Bits ORed into *device_status by the kernels. */
#define SANTA_DEV_BAD_PAGE 1u    /* a page id outside [0, num_pages) */
#define SANTA_DEV_BAD_SEQLEN 2u  /* seq_len < 1 or seq_len > max_teams * team_size */
#define SANTA_DEV_BAD_SEL 4u     /* santa_attend given a sel_ids/sel_count/pi entry out of range */
#define SANTA_DEV_TIMEOUT 8u     /* a bounded wait on an asynchronous copy gave up (2 s) */
#define SANTA_DEV_LAYOUT 16u     /* shared memory not 1 KiB-aligned for the swizzled tile copies;
                                   the kernel returned without writing outputs */

/* Returns SANTA_ABI_VERSION of the loaded library. */
int santa_abi_version(void);

/* Static English text for a santa_status value (never NULL). */
const char* santa_status_string(int status);

/*
 * santa_build_reps — the team representative of every (page, KV head): the mean of the
 * page's valid keys.  [ABS, abstract: each team is represented by one key that the query
 * scores; EXP section 三 step 2 lists the mean key as one choice of representative.]
 *
 *   k_pool      [num_pages][num_kv_heads][team_size][head_dim], dtype.
 *   page_fill   [num_pages] int32 valid-token count of each page (0..team_size), or NULL
 *               for "every page full".  A page with fill 0 gets a zero representative.
 *   reps        [num_pages][num_kv_heads][head_dim] fp32, written.
 *   device_status  one int32 (may be NULL); SANTA_DEV_BAD_SEQLEN if a fill is out of range.
 * Run once after prefill; santa_update_reps refreshes single pages during decode.
 */
int santa_build_reps(const void* k_pool, int dtype, int64_t num_pages, int num_kv_heads,
                     int team_size, int head_dim, const int32_t* page_fill, float* reps,
                     int32_t* device_status, void* stream);

/*
 * santa_update_reps — recompute the representative of the listed pages only (for the pages
 * that received new tokens during decode), with the same arithmetic as santa_build_reps.
 *   pages [num_listed] int32 page ids (device); page_fill as in santa_build_reps (device,
 *   indexed by page id, may be NULL for full pages).  A listed id out of range sets
 *   SANTA_DEV_BAD_PAGE and is skipped.
 */
int santa_update_reps(const void* k_pool, int dtype, int64_t num_pages, int num_kv_heads,
                      int team_size, int head_dim, const int32_t* pages, int num_listed,
                      const int32_t* page_fill, float* reps, int32_t* device_status,
                      void* stream);

/*
 * santa_append_kv — one decode step's new token per (sequence, KV head), written into the
 * paged cache, with the representative of its page brought up to date.  This is the step
 * on either side of the decode path: tokens arrive one at a time and the teams they land in
 * must stay described by their mean key.  [ABS, abstract: one representative key per team;
 * EXP section 三 step 2, mean key; section 八 on keeping teams current as the sequence
 * grows.]
 *
 *   k_new, v_new   [batch][num_kv_heads][head_dim], dtype (device).
 *   seq_lens       [batch] current lengths L_b (device); the token goes to position L_b:
 *                  slot L_b % team_size of page page_table[b][L_b / team_size].
 *   k_pool, v_pool the paged cache, written at that slot.
 *   reps           [num_pages][num_kv_heads][head_dim] fp32; the page's entry becomes the
 *                  mean of its L_b % team_size + 1 valid keys, bit-identical to
 *                  santa_build_reps / santa_update_reps on the grown cache (only that page's
 *                  rows are read).
 *   seq_lens_next  [batch] receives L_b + 1 (may be NULL; must not alias seq_lens).
 *   device_status  SANTA_DEV_BAD_SEQLEN (L_b outside [0, max_teams * team_size)) or
 *                  SANTA_DEV_BAD_PAGE; the sequence is then skipped.
 * The page a token lands in must belong to that sequence alone (a shared-prefix page is
 * never appended to).  Asynchronous on `stream`.
 */
int santa_append_kv(const void* k_new, const void* v_new, int dtype, int batch,
                    int num_kv_heads, int team_size, int head_dim, int max_teams,
                    int64_t num_pages, const int32_t* page_table, const int32_t* seq_lens,
                    void* k_pool, void* v_pool, float* reps, int32_t* seq_lens_next,
                    int32_t* device_status, void* stream);

/* All inputs, outputs and scratch of one decode step (see the layouts above). */
typedef struct santa_decode_args {
  /* inputs */
  const void* q;
  const void* k_pool;
  const void* v_pool;
  const float* reps;           /* read by santa_sample / santa_decode */
  const int32_t* page_table;
  const int32_t* seq_lens;
  int dtype;                   /* santa_dtype of q, k_pool and v_pool */
  int batch;                   /* B */
  int num_q_heads;             /* Hq */
  int num_kv_heads;            /* Hkv, Hq % Hkv == 0 */
  int head_dim;                /* d */
  int team_size;               /* T, also the KV page size */
  int max_teams;               /* row length of page_table */
  int num_draws;               /* M */
  int64_t num_pages;           /* P, rows of k_pool / v_pool / reps */
  uint64_t seed;               /* Philox key */
  /* outputs (santa_attend reads sel_ids, sel_count and pi as inputs) */
  float* out;
  int32_t* draw_ids;
  int32_t* sel_ids;
  int32_t* sel_count;
  float* pi;
  float* team_probs;           /* optional, may be NULL */
  /* scratch: caller-owned device memory (see "Workspace" below), zeroed before first use */
  void* workspace;
  size_t workspace_bytes;
  int32_t* device_status;      /* one int32 the kernels OR SANTA_DEV_* bits into */
  /* sampler variants (santa_sample / santa_decode; zero = the plain method) */
  int32_t sampler;             /* santa_sampler */
  float mix_alpha;             /* defensive mixture weight alpha in [0, 1] */
} santa_decode_args;

/*
 * Samplers.  All draw from q_i = (1 - mix_alpha) p_i + mix_alpha / n, the team distribution
 * with a uniform share mixed in: the defensive mixture of [EXP] section 八 (pitfall 4), which
 * keeps every weight bounded.  mix_alpha = 0 is the plain distribution.  The output pi[k]
 * always holds 1 / (weight of team sel_ids[k]), which santa_attend consumes as it is.
 *   SANTA_SAMPLER_IID_HT      M i.i.d. draws; weight 1/pi_i, pi_i = 1 - (1 - q_i)^M
 *                             (Horvitz-Thompson: the method of [ABS]).
 *   SANTA_SAMPLER_SYSTEMATIC  one uniform u (the Philox word of draw 0), the M points
 *                             (r + u) / M on the CDF; weight 1/pi_i with pi_i = min(1, M q_i)
 *                             (the stratified / systematic variants of [SANTA], abstract).
 *   SANTA_SAMPLER_IID_HH      M i.i.d. draws; weight c_i / (M q_i), c_i the draws of team i
 *                             (Hansen-Hurwitz: the per-draw 1/p_i of [EXP] section 三 step 5).
 * Non-default samplers and mix_alpha > 0 need every unit sampled inside one CTA's shared
 * memory: max_teams <= 1024 and (G + 1) * ceil(max_teams / CL) <= 2048 for the plan's
 * cluster size CL; other shapes return SANTA_ERR_UNSUPPORTED.
 */
typedef enum {
  SANTA_SAMPLER_IID_HT = 0,
  SANTA_SAMPLER_SYSTEMATIC = 1,
  SANTA_SAMPLER_IID_HH = 2
} santa_sampler;

/*
 * Workspace.  A unit is served by one thread-block cluster (up to 16 CTAs sharing their
 * partial results on chip) unless it has so much work that several clusters share it;
 * only then do the clusters' partials and an arrival counter per unit go through the
 * workspace.  santa_decode_workspace_bytes returns the size the library's default plan
 * wants on the current device (0 for an unsupported shape); any size down to
 * santa_decode_workspace_min_bytes also works, with fewer clusters per unit.  When the
 * minimum is 256 bytes (every unit fits one cluster), the workspace may be NULL.  The
 * counters must be zero before the first call (they are left at zero by every call).
 * santa_dense_workspace_bytes sizes the workspace of santa_dense_decode the same way.  A
 * workspace is used by one call at a time.
 */
size_t santa_decode_workspace_bytes(int dtype, int batch, int num_q_heads, int num_kv_heads,
                                    int head_dim, int team_size, int max_teams, int num_draws);
size_t santa_decode_workspace_min_bytes(int batch, int num_q_heads, int num_kv_heads,
                                        int head_dim, int team_size, int max_teams,
                                        int num_draws);

/*
 * santa_sample — score the representatives, form the GQA-mixed team distribution, draw M
 * teams, deduplicate and compute the inclusion probabilities.  Writes draw_ids, sel_ids,
 * sel_count, pi and team_probs (if not NULL).
 * [ABS, abstract: the scores of the representatives decide which teams are sampled; EXP
 * section 三 steps 2-3.]  Uses no workspace.
 */
int santa_sample(const santa_decode_args* a, void* stream);

/*
 * santa_attend — exact attention inside the teams listed in sel_ids[0..sel_count) of every
 * unit, each team weighted by 1/pi, combined as the Horvitz-Thompson ratio into out.
 * sel_ids / sel_count / pi may come from santa_sample or from the caller (distinct team
 * indices < n, any order, pi finite and > 0: the inclusion probability for Horvitz-Thompson
 * weights, M q_i / c_i for Hansen-Hurwitz ones); entries out of range set SANTA_DEV_BAD_SEL
 * and are skipped.
 * [ABS, abstract: attention is exact inside the sampled teams, and each team's share is
 * scaled by one over the probability that the team is in the sample; EXP steps 4-5.]
 */
int santa_attend(const santa_decode_args* a, void* stream);

/*
 * santa_decode_plan — the launch the library would use for `a` (whose pointers need not be
 * valid; only shapes and workspace_bytes are read): out[0] = CTAs per thread-block cluster
 * (CL), out[1] = clusters per unit (NC; NC > 1 routes partials through the workspace),
 * out[2] = teams one CTA scores, out[3] = clusters of CL CTAs the device can run at once,
 * out[4] = 1 if the wide variant runs (bf16 steps whose launch fits one CTA per SM: six
 * stages, two warp groups consuming alternate chunks), else 0.  `out` holds 5 entries.
 * `which`: 0 santa_decode, 1 santa_sample, 2 santa_attend, 3 santa_dense_decode.
 */
int santa_decode_plan(const santa_decode_args* a, int which, int32_t* out);

/* santa_decode — santa_sample followed by santa_attend on `stream`. [ABS] */
int santa_decode(const santa_decode_args* a, void* stream);

/*
 * santa_decode_path — which form of the kernel santa_decode(a) runs (a's pointers need not
 * be valid; shapes, sampler, mix_alpha and workspace_bytes are read).  1: the compact form,
 * for bf16 steps with one cluster per unit and at most 1024 teams per sequence, whose
 * sampling prologue is compiled without the general form's branches (the sampler variants
 * and the mixture run separate instantiations of it); 0: the general form; a negative
 * santa_status for a refused shape.  Both forms compute the same step.
 */
int santa_decode_path(const santa_decode_args* a);

/*
 * santa_dense_decode — exact dense softmax attention over all seq_len tokens of every
 * sequence, split-K over the paged cache (the speed reference the sampled path is compared
 * with; [ABS] compares against a dense FlashAttention baseline).  Reads q, k_pool, v_pool,
 * page_table, seq_lens and the shape fields; writes out; uses workspace and device_status.
 * reps, num_draws, seed and the sampling outputs are ignored.
 */
size_t santa_dense_workspace_bytes(int dtype, int batch, int num_q_heads, int num_kv_heads,
                                   int head_dim, int team_size, int max_teams);
int santa_dense_decode(const santa_decode_args* a, void* stream);

/*
 * santa_decode_noalloc — santa_decode for callers that cannot allocate device memory (no
 * counterpart in the paper; it is a property of this library, not of the method).
 *
 * Who needs it: code that runs where cudaMalloc is not available or not allowed, such as
 * a plug-in inside an inference engine that owns all device memory and lends none after
 * start-up, or a loop that must not allocate once it is running.  Such a caller cannot
 * provide santa_decode's workspace.  This entry point ignores a->workspace and
 * a->workspace_bytes and uses instead a scratch array compiled into the library (a
 * file-scope __device__ array of santa_noalloc_scratch_bytes() = 4 MiB, present on every
 * device that loads the library until the process exits).  It calls no allocator.
 *
 *   - Same inputs, outputs and results as santa_decode (the split plan is the default one
 *     cut down to fit the scratch, so the output may differ from santa_decode's in the
 *     last bits only).
 *   - Returns SANTA_ERR_SCRATCH_LIMIT, before any CUDA call, when the shape needs more than
 *     the scratch holds: santa_decode_workspace_min_bytes > santa_noalloc_scratch_bytes(),
 *     or more than (scratch - 256) / 4 (sequence, KV head) units (their arrival counters).
 *     Every other argument error returns santa_decode's status; a refused call leaves the
 *     array untouched.
 *   - The first call on a device looks up the array's device address (cudaGetSymbolAddress)
 *     with that device current and keeps it for the process; make that first call before any
 *     stream capture.  The kept address is void after cudaDeviceReset on that device (the
 *     module is then loaded again, possibly elsewhere): do not call this entry point after
 *     a reset.
 *   - Every call on a device shares the one array, which keeps the previous call's
 *     contents.  When the plan spreads a unit over several clusters, the call first clears
 *     the arrival counters at the array's start (cudaMemsetAsync on the call's stream, no
 *     allocation).  Calls whose work overlaps on the GPU (different streams, or other
 *     threads) race on the array: serialise them.
 */
int santa_decode_noalloc(const santa_decode_args* a, void* stream);

/*
 * santa_decode_host — one decode step whose inputs come from and whose outputs go to host
 * memory (no counterpart in the paper; a convenience of this library).  On `stream` it
 * copies in_bytes from host_in to dev_in, runs santa_decode(a), copies out_bytes from
 * dev_out to host_out and waits for the stream.
 *
 *   - How each copy is made: when the host buffer is page-locked memory that the current
 *     device reaches at the same address (cudaHostAlloc, a pinned torch tensor) and both
 *     pointers and the size are multiples of 16 bytes, a small kernel of this library moves
 *     the bytes (reading or writing the host memory directly), chained to the decode launch
 *     by programmatic dependent launch; otherwise cudaMemcpyAsync does.  The bytes moved are
 *     the same either way.
 *
 *   - The caller lays out the buffers.  a's input pointers (q, page_table, seq_lens) point
 *     into dev_in, and its output pointers (out, draw_ids, sel_ids, sel_count, pi, and
 *     device_status if the caller wants it back in the same copy) into dev_out, so that
 *     one copy moves each side.  The library reads neither layout: it copies bytes.
 *   - host_in and host_out should be page-locked (cudaHostAlloc or a pinned torch tensor).
 *     Pageable memory works, but then the runtime stages the copies synchronously.
 *   - in_bytes or out_bytes may be 0 (that copy is skipped); otherwise both pointers of
 *     that copy must be non-null (SANTA_ERR_INVALID_ARG, nothing enqueued).
 *   - Returns santa_decode's error if the step is refused (the input copy may already be
 *     enqueued), SANTA_ERR_CUDA if a copy or the stream wait fails, else SANTA_OK after the
 *     host outputs are complete.  device_status is not read here; with device_status in
 *     dev_out, the caller reads the host copy.
 */
int santa_decode_host(const santa_decode_args* a, const void* host_in, void* dev_in,
                      size_t in_bytes, void* host_out, const void* dev_out, size_t out_bytes,
                      void* stream);

/*
 * santa_host_copy_route — how santa_decode_host would move `bytes` between the host buffer
 * `host` and the device buffer `dev` (either direction): 1 when its own copy kernel would
 * (`host` page-locked, reached by the current device at the same address, [host, host +
 * bytes) inside one allocation, both pointers and the size multiples of 16), 0 when
 * cudaMemcpyAsync would (also for null pointers or bytes = 0).  Enqueues nothing.
 */
int santa_host_copy_route(const void* host, const void* dev, size_t bytes);

/*
 * santa_attend_vs — santa_attend with value-row sampling inside every listed team, in place
 * of the full P.V product ([SANTA] "Stochastic Sparse Attention for Memory-Bound
 * Inference", abstract: draw value rows from the post-softmax distribution and gather-add
 * them).  The G query heads of a KV head share one set of S rows per team, drawn from the
 * group-mean in-team softmax r_j; head g weighs a drawn row j by exp(s_gj - m_g) / r_j, and
 * the team denominators stay exact, so the numerator is unbiased given the teams.  Row draw
 * k of team i of unit (b, h) uses Philox4x32-10 word 0 of counter (k, h, b, 1 + i) with key
 * `seed`, decided exactly on a 62-bit fixed-point CDF like the team draws.  Reads only the K
 * rows of the listed teams and S value rows of each.
 *   a          as for santa_attend (sel_ids, sel_count, pi in; out written), num_draws = M
 *              (the slot dimension, <= 1024), seed = key of the row draws, workspace of at
 *              least santa_attend_vs_workspace_bytes bytes (per-team partials).
 *   value_rows S, rows drawn per team, 1..256.
 *   value_ids  [B][Hkv][M][S] int32: the drawn rows (token index within the team), or NULL.
 * Two launches on `stream`.
 */
size_t santa_attend_vs_workspace_bytes(int batch, int num_q_heads, int num_kv_heads,
                                       int head_dim, int num_draws);
int santa_attend_vs(const santa_decode_args* a, int value_rows, int32_t* value_ids,
                    void* stream);

/* Size in bytes of the scratch array santa_decode_noalloc uses. */
size_t santa_noalloc_scratch_bytes(void);

#ifdef __cplusplus
}
#endif

#endif /* SANTA_H */
