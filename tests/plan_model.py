"""The launch shape the split-count heuristic is fed, written out for the
tests (no CUDA, no library calls): how many CTAs a split takes and how many
the GPU holds at once.

"Flash-Decoding: Split-KV Attention for Long-Context Decode", §6 "How many
splits?" plans over work items (one per CTA of a split) and slots (CTAs that
run at once; its dispatcher passes two per SM).  With grouped heads one CTA
serves a KV head's whole group (§1 GQA note), so work = batch x KV heads for
up to 16 (position, head) columns.  The readings for wider groups: the
tcgen05 CTA of 17-128 columns (16-bit cache, tensor cores) still serves all
of them but takes a whole SM, so it has one slot per SM; past that (or on an
fp8 cache or the CUDA cores) a split takes one CTA per 16 columns."""


def slot_model(B, Hkv, G, q_len, fp8, cuda_cores, sms):
    """(work items, slots) of one split-kernel launch."""
    cols = G * q_len
    if cols <= 16:
        return B * Hkv, 2 * sms
    if cols <= 128 and not fp8 and not cuda_cores:
        return B * Hkv, sms
    return B * Hkv * -(-cols // 16), 2 * sms
