/*
 * Plain, slow, single-threaded CPU oracle for the reduce-copy and batched-copy
 * path.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the bench's
 * CPU-baseline leg may load it; the product path never does.  It shares no
 * code, header, table or constant generator with the CUDA library.
 *
 * Every function restates one passage of the pages it follows:
 *   [TBV]  "TransferBench data validation" (ROCm docs 1.66.02)
 *            - table "Number of sources / Expected value"
 *            - section "Expected source pattern"
 *            - section "Expected destination (dstReference)"
 *            - section "How validation (ValidateAllTransfers) works"
 *   [ROT]  TransferBench PR #365 "Fix one-sided remote-read bandwidth inflation
 *          via source-slice rotation (SRC_ROTATE_BYTES)", section
 *          "Technical Details" (the K rule, allocation and folding bullets)
 *   [MC]   Mooncake RFC #5041 "HipTransport: fast, correct intra-node XGMI",
 *          section "Design of #5040": a (src, dst, len) descriptor array
 *   [SM64] Steele, Lea, Flood, "Fast splittable pseudorandom number
 *          generators", OOPSLA 2014 (SplitMix64), used where the pages leave
 *          fillCompress's random source unnamed.
 *
 * Build: gcc -O2 -std=c99 -ffp-contract=off -fno-fast-math (no FMA contraction,
 * no reassociation, subnormals kept), so each float add below is one IEEE-754
 * binary32 round-to-nearest-even addition.
 *
 * Parity status: the pages name fillCompress's 1B0/2B0/4B0/32B0 modes without
 * defining them, so orc_fill_compress follows a stated reading (below).  That
 * reading is pinned by hand-worked words (tests/golden/fill_compress.txt,
 * derived with integer arithmetic from the published SplitMix64 vector), which
 * fix its draw order, float mapping, each zero mask, the mode boundary, the
 * partial last line and the per-buffer seed.
 */
#include <stdint.h>
#include <stddef.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* [TBV] "Expected source pattern", Default row:                           */
/*   PrepSrcValue(bufferIdx, i) = (((i % 383) * 517) % 383 + 31) * (bufferIdx + 1) */
/* i is the element index inside the transfer; the integer result is stored */
/* as a float32 (every value is at most 413 * (bufferIdx + 1), exact).      */
/* ------------------------------------------------------------------------ */
float orc_prep_src_value(int64_t bufferIdx, uint64_t i)
{
    uint64_t v = (((i % 383u) * 517u) % 383u + 31u) * (uint64_t)(bufferIdx + 1);
    return (float)v;
}

void orc_prepare_reference_default(float *out, uint64_t n, int64_t bufferIdx)
{
    for (uint64_t i = 0; i < n; ++i)
        out[i] = orc_prep_src_value(bufferIdx, i);
}

/* ------------------------------------------------------------------------ */
/* [TBV] "Expected source pattern", fillPattern row: the given vector of    */
/* floats repeated over the buffer.                                         */
/* ------------------------------------------------------------------------ */
void orc_fill_pattern(float *out, uint64_t n, const float *pattern, uint64_t patLen)
{
    for (uint64_t i = 0; i < n; ++i)
        out[i] = pattern[i % patLen];
}

/* ------------------------------------------------------------------------ */
/* [SM64] SplitMix64, sequential form: the state advances by the golden     */
/* gamma, then the 64-bit finaliser mixes it.                               */
/* ------------------------------------------------------------------------ */
uint64_t orc_splitmix64_next(uint64_t *state)
{
    uint64_t z;
    *state += 0x9E3779B97F4A7C15ull;
    z = *state;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

void orc_splitmix64_stream(uint64_t seed, uint64_t *out, uint64_t count)
{
    uint64_t s = seed;
    for (uint64_t j = 0; j < count; ++j)
        out[j] = orc_splitmix64_next(&s);
}

/* ------------------------------------------------------------------------ */
/* [TBV] "Expected source pattern", fillCompress row: random floats with    */
/* optional zeroing per 64-byte line; mode 0 = random, 1 = 1B0, 2 = 2B0,    */
/* 3 = 4B0, 4 = 32B0; percentages control the mix.                           */
/*                                                                          */
/* Reading taken (the page defines neither the masks nor the draw):        */
/*  - a line is 16 floats; buffer k uses the SplitMix64 stream seeded with  */
/*    seed + k, read sequentially: per line one draw picks the mode, then   */
/*    16 draws give the floats (all 16 always drawn);                        */
/*  - mode = first m with (draw % 100) < pct[0] + ... + pct[m];             */
/*  - float = (draw >> 40) * 2^-23 - 1, exact, in [-1, 1);                   */
/*  - mode "nB0" zeroes every odd-numbered aligned n-byte chunk of the line */
/*    (1B0: bytes 1,3,..,63; 2B0: bytes 2-3,6-7,..; 4B0: floats 1,3,..,15;  */
/*    32B0: bytes 32..63).  Bytes are in memory (little-endian) order.      */
/* A partial last line keeps only its first (n % 16) floats.                */
/* Returns 0, or -1 when the percentages do not sum to 100.                 */
/* ------------------------------------------------------------------------ */
static const unsigned orc_zero_chunk_bytes[5] = { 0u, 1u, 2u, 4u, 32u };

int orc_fill_compress(float *out, uint64_t n, const uint32_t pct[5], uint64_t seed,
                      int64_t bufferIdx)
{
    uint32_t cum[5];
    uint32_t total = 0;
    for (int m = 0; m < 5; ++m) {
        total += pct[m];
        cum[m] = total;
    }
    if (total != 100u)
        return -1;

    uint64_t state = seed + (uint64_t)bufferIdx;
    uint64_t nLines = (n + 15u) / 16u;
    for (uint64_t line = 0; line < nLines; ++line) {
        uint64_t r = orc_splitmix64_next(&state) % 100u;
        int mode = 0;
        while (mode < 4 && r >= cum[mode])
            ++mode;

        float vals[16];
        for (int j = 0; j < 16; ++j) {
            uint64_t d = orc_splitmix64_next(&state);
            vals[j] = (float)(int32_t)(d >> 40) * 0x1p-23f - 1.0f;
        }

        unsigned char bytes[64];
        memcpy(bytes, vals, 64);
        unsigned chunk = orc_zero_chunk_bytes[mode];
        if (chunk != 0u) {
            for (unsigned b = 0; b < 64u; ++b) {
                if ((b / chunk) % 2u == 1u)
                    bytes[b] = 0;
            }
        }
        memcpy(vals, bytes, 64);

        for (int j = 0; j < 16; ++j) {
            uint64_t i = line * 16u + (uint64_t)j;
            if (i < n)
                out[i] = vals[j];
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* [TBV] "Expected destination (dstReference)":                             */
/*   dstReference[0] = memset to MEMSET_CHAR                                */
/*   dstReference[1] = srcReference[0]                                      */
/*   dstReference[k] = dstReference[k-1] + srcReference[k-1]                */
/* and dstReference[numSrcs] is the expected result.  out holds the running */
/* dstReference[k], advanced one k at a time, and ends as                   */
/* dstReference[nSrc].  Step 1 copies bytes (1 source: dst == src0, bit for */
/* bit); every later step is one float32 add per element.                   */
/* ------------------------------------------------------------------------ */
void orc_dst_reference(const float *const *srcRef, int nSrc, uint64_t n,
                       uint8_t memsetByte, float *out)
{
    if (nSrc == 0) {
        memset(out, memsetByte, (size_t)(n * sizeof(float)));
        return;
    }
    memcpy(out, srcRef[0], (size_t)(n * sizeof(float)));
    for (int k = 2; k <= nSrc; ++k) {
        const float *src = srcRef[k - 1];
        for (uint64_t i = 0; i < n; ++i)
            out[i] = out[i] + src[i];
    }
}

/* ------------------------------------------------------------------------ */
/* [ROT] "Technical Details":                                               */
/*   K = ceil(SRC_ROTATE_BYTES / numBytes), default 256MB, 0 disables       */
/*   allocation = K * numBytes + byteOffset                                 */
/* 0 = disabled means K = 1.  Slice j starts at j * stride, with the stride */
/* numBytes rounded up to 256 bytes (the review asks for slices aligned for */
/* vector loads), and the allocation ends right after the last slice:       */
/* (K - 1) * stride + numBytes + byteOffset, which is the page's            */
/* K * numBytes + byteOffset whenever numBytes is a multiple of 256.        */
/* Returns 0, or -1 for numBytes == 0 or a 64-bit overflow.                 */
/* ------------------------------------------------------------------------ */
int orc_rotation_plan(uint64_t numBytes, uint64_t rotateBytes, uint64_t byteOffset,
                      uint64_t *K, uint64_t *sliceStride, uint64_t *allocBytes)
{
    if (numBytes == 0 || numBytes > UINT64_MAX - 255u)
        return -1;
    uint64_t k = 1;
    if (rotateBytes != 0) {
        k = rotateBytes / numBytes;
        if (rotateBytes % numBytes != 0)
            k += 1;
    }
    uint64_t stride = (numBytes + 255u) / 256u * 256u;
    if (k - 1 > (UINT64_MAX - numBytes) / stride)
        return -1;
    uint64_t alloc = (k - 1) * stride + numBytes;
    if (alloc > UINT64_MAX - byteOffset)
        return -1;
    *K = k;
    *sliceStride = stride;
    *allocBytes = alloc + byteOffset;
    return 0;
}

/* [ROT] "RotateSourceSlices()": iteration i reads slice i % K, with the    */
/* iteration folded into [0, K) so negative warm-up indices work.           */
uint64_t orc_slice_for_iteration(int64_t iteration, uint64_t K)
{
    int64_t k = (int64_t)K;
    int64_t r = iteration % k;
    if (r < 0)
        r += k;
    return (uint64_t)r;
}

/* ------------------------------------------------------------------------ */
/* [MC] "Design of #5040": one launch over a (src, dst, len) descriptor     */
/* array; each descriptor is a plain memcpy.  Here src and dst are byte     */
/* offsets into two host pools.  Returns 0, or -1 (nothing further copied)  */
/* at the first descriptor that falls outside its pool.                     */
/* ------------------------------------------------------------------------ */
int orc_apply_batch(uint8_t *dstPool, uint64_t dstPoolBytes,
                    const uint8_t *srcPool, uint64_t srcPoolBytes,
                    const uint64_t *srcOff, const uint64_t *dstOff,
                    const uint64_t *len, uint64_t n)
{
    for (uint64_t d = 0; d < n; ++d) {
        if (srcOff[d] > srcPoolBytes || len[d] > srcPoolBytes - srcOff[d])
            return -1;
        if (dstOff[d] > dstPoolBytes || len[d] > dstPoolBytes - dstOff[d])
            return -1;
        memcpy(dstPool + dstOff[d], srcPool + srcOff[d], (size_t)len[d]);
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* [TBV] "How validation (ValidateAllTransfers) works", step 3: memcmp of   */
/* output against expected; on mismatch, find the first differing index.   */
/* Returns the first differing element index (elements of elemSize bytes),  */
/* or -1 when the buffers are equal.                                        */
/* ------------------------------------------------------------------------ */
int64_t orc_first_mismatch(const void *actual, const void *expected,
                           uint64_t nBytes, uint64_t elemSize)
{
    if (memcmp(actual, expected, (size_t)nBytes) == 0)
        return -1;
    const unsigned char *a = (const unsigned char *)actual;
    const unsigned char *e = (const unsigned char *)expected;
    for (uint64_t b = 0; b < nBytes; ++b) {
        if (a[b] != e[b])
            return (int64_t)(b / elemSize);
    }
    return -1;
}
