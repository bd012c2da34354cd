"""Float64 CPU oracle for the KDA core recurrence.

TEST INFRASTRUCTURE ONLY: imported by tests/, by the smoke check and by the
benchmark's CPU-baseline / reference leg; never by the library itself.
"""
