"""Prints the library's kernel budget table.

    python -m bit_quantized_tensor_gb300.budget            # host only
    python -m bit_quantized_tensor_gb300.budget --measure  # + registers and residency (needs a GPU)

One row per kernel instance: threads, dynamic shared memory, tensor-memory
columns, cluster size and the CTAs per SM the design counts on; with
--measure also the registers per thread, static shared memory and the CTAs
per SM the device's occupancy calculator allows at that launch shape.
"""
import argparse

import bit_quantized_tensor_gb300 as qg

# Per-SM limits of sm_103a: shared memory an SM can give its CTAs (228 KiB,
# of which each CTA also takes 1 KiB for the system), tensor-memory columns.
SM_SMEM_BYTES = 233472
CTA_RESERVED_SMEM = 1024
CTA_SMEM_LIMIT = 232448
TMEM_COLUMNS = 512
MAX_THREADS_PER_CTA = 1024
MAX_PORTABLE_CLUSTER = 8


def accounting_errors(entry: dict) -> list:
    """What is wrong with one entry's budget on the host side (empty when it
    fits): shared memory per CTA and per SM at the design residency, tensor
    memory per SM, threads per CTA, cluster size."""
    e, errs = entry, []
    ctas = e["min_ctas_per_sm"]
    if e["smem_bytes"] > CTA_SMEM_LIMIT:
        errs.append(f"{e['smem_bytes']} B dynamic shared memory > {CTA_SMEM_LIMIT} per CTA")
    if ctas * (e["smem_bytes"] + CTA_RESERVED_SMEM) > SM_SMEM_BYTES:
        errs.append(f"{ctas} CTAs x {e['smem_bytes']} B do not fit the SM's shared memory")
    if e["tmem_cols"] and (e["tmem_cols"] not in (32, 64, 128, 256, 512) or ctas * e["tmem_cols"] > TMEM_COLUMNS):
        errs.append(f"{ctas} CTAs x {e['tmem_cols']} tensor-memory columns do not fit {TMEM_COLUMNS}")
    if not 32 <= e["threads"] <= MAX_THREADS_PER_CTA or e["threads"] % 32:
        errs.append(f"{e['threads']} threads per CTA")
    if not 1 <= e["cluster"] <= MAX_PORTABLE_CLUSTER:
        errs.append(f"cluster of {e['cluster']}")
    if ctas < 1:
        errs.append("needs no resident CTA")
    return errs


def format_table(rows: list) -> str:
    cols = ["kernel", "threads", "smem_bytes", "tmem_cols", "cluster", "min_ctas_per_sm"]
    if rows and "ctas_per_sm" in rows[0]:
        cols += ["regs_per_thread", "static_smem_bytes", "ctas_per_sm"]
    width = {c: max(len(c), *(len(str(r[c])) for r in rows)) for c in cols}
    lines = ["  ".join(c.ljust(width[c]) for c in cols)]
    lines += ["  ".join(str(r[c]).ljust(width[c]) for c in cols) for r in rows]
    return "\n".join(lines)


def main() -> None:
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--measure", action="store_true", help="add registers and residency (needs a GPU)")
    args = ap.parse_args()
    rows = qg.kernel_budgets(measure=args.measure)
    print(format_table(rows))
    bad = [(r["kernel"], accounting_errors(r)) for r in rows if accounting_errors(r)]
    for name, errs in bad:
        print(f"BUDGET {name}: " + "; ".join(errs))
    raise SystemExit(1 if bad else 0)


if __name__ == "__main__":
    main()
