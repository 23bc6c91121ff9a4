"""Counts gathered by the BF16 parity checks, printed at the end of the test
session: how many outputs matched within one BF16 ulp of the correctly
rounded exact value, and how many needed the cancellation clause
(|y - y*| <= 1e-5 * T + ulp/2) instead."""
BF16 = {"checked": 0, "within_1ulp": 0, "by_cancellation_clause": 0}


def record_bf16(n_checked: int, n_ulp: int, n_clause_only: int) -> None:
    BF16["checked"] += int(n_checked)
    BF16["within_1ulp"] += int(n_ulp)
    BF16["by_cancellation_clause"] += int(n_clause_only)
