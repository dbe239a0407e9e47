"""Reporting conventions of the pages (host-side arithmetic on measured numbers).

* Acceptance length counts the bonus token: the number of tokens a verification
  round completes is n + 1 ("SpecOPD" summary (onedev.kr), section "premises and
  limits"; the ABI returns n, the drafts accepted).
* Cycle cost c = L / S: acceptance length over the throughput multiple against
  autoregressive decoding, i.e. how many autoregressive-token times one draft/verify
  cycle takes ("DSpine card numbers and public file headers" (aiwithghost.com),
  section on the ten cells of the card).
* Speedup = new throughput / baseline throughput.
"""


def acceptance_length(n_accepted):
    """Mean tokens completed per verification round (bonus included)."""
    n = [int(x) for x in n_accepted if int(x) >= 0]
    if not n:
        return float("nan")
    return sum(x + 1 for x in n) / len(n)


def cycle_cost(acceptance_len, throughput, throughput_ar):
    """c = L / S with S = throughput / throughput_ar."""
    return acceptance_len / (throughput / throughput_ar)


def speedup(throughput, throughput_base):
    return throughput / throughput_base


def gain_pct(new, old):
    return (new / old - 1.0) * 100.0
