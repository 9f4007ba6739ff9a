"""CPU oracle of the DFlash draft + verify step (test infrastructure only).

Only tests, the package smoke check and the benchmark's CPU-baseline leg may import it.
"""
