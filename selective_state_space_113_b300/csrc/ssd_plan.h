// ssd_plan.h -- which walk the tensor-core SSD kernels take for a problem, and
// how the ticket walk cuts the heads (host only; no CUDA).
//
// One head per CTA (the block scheduler hands heads to SMs as they free up)
// unless that leaves the last wave mostly empty: the waves, rounded up, more
// than 15% above the heads' share of the SMs, as 320 heads on 148 SMs (2.16
// waves, run as 3).  Then the ticket walk, with each head cut into equal
// segments of about a sixth of a CTA's share of the chunks.  Measured on the
// Mamba-2 2.7B-shaped layer (32 chunks per head, 69 per CTA), on one box:
// segments of 2, 3, 4, 5, 8, 11, 16, 32 chunks took 0.389, 0.353, 0.337,
// 0.327, 0.324, 0.313, 0.326, 0.376 ms; on another, 5, 8 and 11 took 0.330,
// 0.325 and 0.325 -- each unit costs about 3 us of hand-off and restart, and
// the tail is up to a unit.
#pragma once

namespace ssm {
namespace ssdtc {

struct Plan {
    bool dyn;         // the ticket walk
    long long seg;    // chunks per segment (the whole head when !dyn)
    long long nseg;   // segments per head
    long long units;  // heads x segments
    long long ctas;   // CTAs launched
};

// heads = batch x H, nch = chunks per head, sms = the GPU's SMs (one CTA each).
// want_seg > 0 or want_ctas > 0 (development and tests) ask for the ticket
// walk with segments of that many chunks and at most that many CTAs.
inline Plan plan(long long heads, long long nch, long long sms, long long want_seg = 0,
                 long long want_ctas = 0) {
    Plan p;
    const long long waves = (heads + sms - 1) / sms;
    p.dyn = (heads > sms && waves * sms * 100 > heads * 115) || want_seg > 0 || want_ctas > 0;
    p.seg = nch;
    if (p.dyn) {
        const long long share = heads * nch / sms;   // chunks per CTA
        long long n = share > 0 ? (6 * nch + share - 1) / share : 1;
        if (n < 1) n = 1;
        if (n > nch) n = nch;
        p.seg = (nch + n - 1) / n;
        if (want_seg > 0) p.seg = want_seg < nch ? want_seg : nch;
    }
    p.nseg = (nch + p.seg - 1) / p.seg;
    p.units = heads * p.nseg;
    p.ctas = p.dyn ? (p.units < sms ? p.units : sms) : heads;
    if (want_ctas > 0 && want_ctas < p.ctas) p.ctas = want_ctas;
    return p;
}

}  // namespace ssdtc
}  // namespace ssm
